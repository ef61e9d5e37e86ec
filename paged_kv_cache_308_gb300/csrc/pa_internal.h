// Internal interface between the C-ABI layer (pa_api.cpp) and the decode
// kernels (pa_kernels.cu).  Not installed; the public interface is
// include/pa_decode.h.  The chunked-prefill kernels have their own (pa_prefix.h).
#pragma once

#include <cuda.h>          // CUtensorMap (header only; the driver is reached at run time)
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>

namespace pa {

constexpr int kBlockSize = 16;    // tokens per KV block (one MMA M-tile of tokens)
constexpr int kMaxGroup = 8;      // query heads per kv head: the MMA N dimension
constexpr int kReduceThreads = 256;
constexpr int kReduceMinSlice = 32;  // narrowest head_dim slice of a reduce CTA
constexpr unsigned kDefaultWaitLimit = 1u << 20;

// Partition size of a sequence of L tokens in the persistent schedule with a
// given partition size `pmax`: the fewest partitions of at most pmax tokens,
// evened out and rounded up to whole blocks (so every partition is
// non-empty).  The partition count is (L + size - 1) / size.
__host__ __device__ inline int balanced_partition(int L, int pmax) {
    if (L <= 0) return pmax;
    const int n = (L + pmax - 1) / pmax;
    const int even = (L + n - 1) / n;
    return ((even + kBlockSize - 1) / kBlockSize) * kBlockSize;
}

// Pooled split (PA_FLAG_POOLED): the blocks of a (sequence, kv head) are
// dealt to the warps of its partition CTAs in chunks of pool_chunk(stages)
// blocks (at least the copy depth, so the copies run at most one chunk
// ahead); each warp takes three chunks round-robin and claims the rest from
// a 64-bit counter whose high word must read kClaimTag (the reduce kernel
// writes kClaimTag << 32 after every call).  Any other value -- a workspace
// never used by a pooled call -- keeps every warp on the round-robin, which
// needs no counter.  Every CTA has a chunk when the partition size is at
// least warps * chunk * kBlockSize tokens.
constexpr int kPoolChunk = 2;
constexpr unsigned kClaimTag = 0x5a17c0deu;
__host__ __device__ constexpr int pool_chunk(int stages) { return stages > kPoolChunk ? stages : kPoolChunk; }
inline int pool_min_partition(int warps, int stages) { return warps * pool_chunk(stages) * kBlockSize; }

// Batches of at most this many sequences keep the persistent schedule's work
// list, order, lengths and partition sizes in each CTA's shared memory (these
// extra bytes).
constexpr int kPersistentSeqCache = 256;
constexpr int persistent_seq_cache_bytes(int num_seqs) {
    return num_seqs <= kPersistentSeqCache ? ((4 * num_seqs + 1) * 4 + 15) / 16 * 16 : 0;
}

// Runs `set` (a kernel's launch attributes, which are per device) the first
// time it is reached on each device, tracked in that kernel's `done` word
// (one bit per device; devices past 63 set it every time).  Each attribute
// call costs driver time that a short decode call would notice.
template <typename F>
inline cudaError_t once_per_device(std::atomic<unsigned long long>& done, F&& set) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = set();
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

struct PartitionParams {
    __half* out;
    const __half* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    float* max_logits;  // [B][H][max_partitions], log2 domain
    float* exp_sums;    // [B][H][max_partitions]
    float* tmp_out;     // [B][H][max_partitions][D], normalised partial outputs
    long long num_blocks;
    int num_heads, num_kv_heads, group;
    int max_blocks_per_seq, max_seq_len;
    int partition_size, max_partitions;
    float scale_log2;   // scale * log2(e)
    unsigned wait_limit;
    int force_timeout;
    // Diagnostic builds (-DPA_TRACE) only: per-CTA records of
    // {sm id, entry, first block ready, main loop done, exit} in globaltimer ns.
    unsigned long long* trace;
    // Fused combine: two words per (sequence, kv head) (the ticket or the
    // arrivals, then the departures), zero before the call and left zero
    // after it; null when a separate reduce kernel merges.
    unsigned int* tickets;
    // Persistent schedule: the sequences in schedule order (seq_order), the
    // exclusive prefix sums of their work items in that order (num_seqs + 1
    // entries), each sequence's partition size, and the next item to hand
    // out; null for one CTA per grid cell.
    const int* work_offsets;
    const int* seq_order;
    const int* part_sizes;
    int* work_counter;
    int num_seqs;
    // Device status word (PA_DEV_* bits) for kernels compiled outside
    // pa_kernels.cu, where the word itself is defined.
    unsigned int* status;
    // Pooled split: one claim counter per (sequence, kv head); null for the
    // fixed assignment of blocks to partitions.
    unsigned long long* claims;
    // Partials of a range of partitions (split-KV across devices): CTA x
    // computes partition part_begin + x of its sequence and always writes a
    // partial (slot x of max_partitions), never the output; a partition past
    // the sequence's end gets the empty partial (m = -inf, l = 0, acc = 0).
    int part_begin = 0;
    int partials_only = 0;
    // Flat one-wave split (persistent kernel without a work list; flat = 1):
    // max_partitions is then the CTAs per kv head, and part_counts receives
    // the number of partials of each sequence from the CTA that holds its
    // first block (null when there is one CTA per kv head: no partials).
    int flat = 0;
    int* part_counts = nullptr;
    // Fused combine on a co-resident (cooperatively launched) grid: the CTAs
    // of a (sequence, kv head) meet at a group barrier and merge in parallel
    // (tickets then holds an arrival and a departure word per group).
    int coop = 0;
};

struct ReduceParams {
    __half* out;
    const float* max_logits;
    const float* exp_sums;
    const float* tmp_out;
    const int32_t* seq_lens;
    int num_heads, max_blocks_per_seq, max_seq_len;
    int partition_size, max_partitions;
    const int* part_sizes;  // per-sequence partition sizes (persistent schedule), else null
    // Pooled split: the claim counters to re-arm (kClaimTag << 32), one per
    // (sequence, kv head); null otherwise.
    unsigned long long* claims;
    int group;  // query heads per kv head
    // Merge of partials gathered from several sources (split-KV across
    // devices): partition p of a sequence is slot p % src_parts of source
    // p / src_parts, the sources src_stride rows apart; every sequence's
    // output is written (one partial, or none for an empty sequence, too).
    // src_parts = 0: the partials of one partition grid (max_partitions
    // slots per (sequence, head)), and sequences with at most one partition
    // are skipped.
    int src_parts = 0;
    long long src_stride = 0;
    // Flat split: the number of partials of each sequence (else derived from
    // the partition size)
    const int* part_counts = nullptr;
};

struct ScanParams {
    const int32_t* seq_lens;
    int* work_offsets;  // [num_seqs + 1], over the schedule order
    int* seq_order;     // [num_seqs]: schedule position -> sequence
    int* part_sizes;    // [num_seqs]: partition size of each sequence
    int* work_counter;  // set to first_dynamic (the persistent grid size)
    int num_seqs, max_seq_len, max_blocks_per_seq, num_kv_heads, first_dynamic;
    int partition_size;  // > 0: balanced_partition with this size
    int slots;           // else partitions per kv head to apportion (the cap that fits them)
};

// Dynamic shared memory of a partition CTA of `warps` warps with `stages`
// stages each (includes 1 KB of alignment slack for the 128-byte swizzle);
// -1 for a shape that is not compiled.
int partition_smem_bytes(int head_dim, int warps, int stages);

// prm.claims selects the pooled form of the kernel.  With prm.coop the grid
// is launched cooperatively (every CTA resident at once); a grid larger than
// the device holds at once returns cudaErrorCooperativeLaunchTooLarge without
// launching anything.
cudaError_t launch_partition(int head_dim, int warps, int stages, const PartitionParams& prm,
                             const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, dim3 grid, cudaStream_t stream);

// Bytes of the stage area the fused combine's parallel merge needs for n
// partitions of a group of `group` heads (defined in pa_kernels.cu).
long long fused_barrier_bytes(int n, int group, int head_dim);

// Both kernels are launched as programmatic dependents of the preceding work
// on the stream, so their start-up overlaps its tail; each waits on the
// dependency before it reads any memory.  `width` is the head_dim slice of a
// reduce CTA (32, 64, 128 or 256, at most head_dim).
cudaError_t launch_reduce(int head_dim, int width, const ReduceParams& prm, dim3 grid, cudaStream_t stream);

// The disarmed state of the pooled split's claim counters (all zero, so the
// next pooled call deals its chunks round-robin), for a call whose reduce
// launch failed after its partition launch had consumed claims.
cudaError_t disarm_claims(unsigned long long* claims, size_t count, cudaStream_t stream);

// The persistent schedule's work list: one CTA sizes the partitions, orders the
// sequences longest partition first and sums their item counts.
cudaError_t launch_work_scan(const ScanParams& prm, cudaStream_t stream);

// Persistent schedule: `grid` CTAs of `warps` warps take the items of the
// work list in prm.work_offsets from prm.work_counter; persistent_smem_bytes
// is the dynamic shared memory of one such CTA (-1 for a shape that is not
// compiled).
int persistent_smem_bytes(int head_dim, int warps, int stages);
cudaError_t launch_partition_persistent(int head_dim, int warps, int stages, const PartitionParams& prm,
                                        const CUtensorMap& tk, const CUtensorMap& tv, int grid, cudaStream_t stream);

// Read and clear the status word of the current device (synchronises stream).
cudaError_t read_and_clear_status(cudaStream_t stream, int* status);

// Device address of that status word on the current device (null on error);
// kernels of other translation units record their errors through it.
unsigned int* device_status_ptr();

}  // namespace pa
