// Internal interface between the C-ABI layer (pa_api.cpp) and the
// chunked-prefill kernels (pa_prefix.cu).  Not installed.
#pragma once

#include "pa_internal.h"

namespace pa {

struct PrefixParams {
    __half* out;                    // [num_tokens][H][D]
    const __half* q;                // [num_tokens][H][D]
    const int32_t* block_tables;    // context blocks
    const int32_t* context_lens;    // [B]
    const int32_t* query_start_loc; // [B + 1]
    long long num_blocks;
    int num_heads, num_kv_heads, group;
    int max_blocks_per_seq, max_context_len, max_query_len, num_tokens;
    float scale_log2;
    unsigned wait_limit;
    int force_timeout;
    unsigned int* status;           // device status word (PA_DEV_* bits are OR-ed in)
    // Key split of the last wave (tcgen05 kernel; split_parts == 0: off, and
    // the grid is (query tiles, kv heads, sequences)).  Otherwise the grid is
    // 1-D over units numbered as that grid's CTAs (tile fastest, then kv head,
    // then sequence; tiles_per_seq tiles per kv head): CTAs [0, split_whole)
    // run units [0, split_whole) whole, and CTA split_whole + r * split_parts + p
    // runs part p of the key tiles of unit split_whole + r, leaving its rows'
    // unnormalised partial in split_o / split_ml for pa_prefix_merge_kernel.
    int split_whole = 0;
    int split_parts = 0;
    int tiles_per_seq = 0;
    float* split_o = nullptr;       // [R][split_parts][128 rows][D]: O relative to 2^m
    float* split_ml = nullptr;      // [R][split_parts][128 rows][2]: m (scaled, log2), l
    // Persistent form of the tcgen05 kernel (sched != nullptr): a fixed grid
    // whose CTAs claim the total_units units (numbered as the CTAs above,
    // tiles_per_seq set in either form) from the counter sched[0]; sched[1]
    // counts the CTAs that finished, and the last one re-arms both to zero.
    unsigned int* sched = nullptr;
    int total_units = 0;
    // Diagnostic builds (-DPA_TRACE) only: the tcgen05 kernel records
    // SM clock stamps of its pipeline events, kPrefixTraceIters x 16 per CTA
    // (the last of the kPrefixTraceIters records holds the CTA's phases in
    // global-timer ns).
    unsigned long long* trace;
};

constexpr int kPrefixTraceIters = 256;

// Chunked-prefill kernel: grid (query tiles, kv heads, sequences); maps are
// {K cache, V cache (2-D, as for decode), K new, V new (3-D [token][kv head][dim])}.
int prefix_smem_bytes(int head_dim);
cudaError_t launch_prefix(int head_dim, const PrefixParams& prm, const CUtensorMap* maps, dim3 grid,
                          cudaStream_t stream);
// The tcgen05 version: 128-row tiles (floor(128 / G) tokens); its V maps are
// whole-block views (3-D cache, 4-D chunk) whose box is one block.
int prefix_tc_smem_bytes(int head_dim);
// CTAs of the tcgen05 kernel one SM holds at once (shared and tensor memory, registers).
int prefix_tc_ctas_per_sm(int head_dim);
cudaError_t launch_prefix_tc(int head_dim, const PrefixParams& prm, const CUtensorMap* maps, dim3 grid,
                             cudaStream_t stream);
// Rows rounded up by the tcgen05 kernel's tiles (the MMA M), for the split workspace.
constexpr int kPrefixTileRows = 128;
// The merge of a key split: the fp16 output rows of its `units` split units
// from their parts' partials (a programmatic dependent of the tcgen05 kernel).
cudaError_t launch_prefix_merge(int head_dim, const PrefixParams& prm, int units, cudaStream_t stream);

}  // namespace pa
