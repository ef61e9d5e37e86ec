// pa_decode_noalloc: the decode call for callers that must not allocate
// device memory.
//
// Some callers cannot call cudaMalloc.
// - A framework or serving engine may own all device memory through its own
//   pool; an allocation behind its back can fail, or upset its accounting.
// - A latency-critical decode loop cannot afford the synchronisation that a
//   first-time or growing allocation brings.
// - Code running from a host callback may not call allocating CUDA functions
//   at all.
// pa_decode grows a cached workspace with cudaMalloc, and pa_decode_ex wants
// the caller to hand it one.  This entry point needs neither.  The split-KV
// partials live in the file-scope device array below, whose fixed size every
// GPU that loads this library holds until the process exits.
#include <mutex>

#include "pa_decode.h"
#include "pa_internal.h"

// Scratch shared by every call of pa_decode_noalloc on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices];

// In host code `g_noalloc_scratch` names a host-side stand-in, not the device
// array, so the device address is looked up once per device, with that
// device current, and then reused.
int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return PA_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                                 int max_blocks_per_seq, int max_seq_len, int64_t num_blocks, int num_heads,
                                 int num_kv_heads, int head_dim, int block_size, float scale, pa_stream_t stream) {
    pa_decode_args a;
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.num_seqs = num_seqs;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.max_seq_len = max_seq_len;
    a.num_blocks = num_blocks;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.scale = scale;
    pa_decode_plan_t plan;
    int rc = pa_decode_plan(&a, nullptr, 0, &plan);
    if (rc) return rc;
    if (plan.workspace_bytes > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    void* ws = nullptr;
    if (plan.workspace_bytes > 0) {
        rc = noalloc_scratch(&ws);
        if (rc) return rc;
    }
    // Every partial the reduce reads is written earlier in the same call, and
    // the pooled plan's claim counters treat anything but their own armed
    // state (which the reduce leaves behind) as "not armed"; so nothing in the
    // scratch has to start at zero, whatever shape the previous call had.
    return pa_decode_ex(&a, nullptr, ws, plan.workspace_bytes > 0 ? PA_NOALLOC_SCRATCH_BYTES : 0, stream);
}
