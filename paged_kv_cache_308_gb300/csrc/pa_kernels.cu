// Split-KV paged-attention decode kernels for GB300 (sm_103a).
//
// pa_partition_kernel -- Phase 1 of the "docs" commit page (partition kernel
//   gridded on kv heads): one CTA per (partition, kv head, sequence).  Every
//   K/V block of the partition is fetched once from HBM by TMA and used by
//   all query heads of the GQA group.  It writes the compound partial
//   (max score, exp sum, normalised weighted V) of the "docs" commit page, or
//   the final output when the sequence has a single partition.
// pa_partition_persistent_kernel -- the same partition work over a fixed grid
//   of one-warp CTAs that walk a device-built work list (PA_MODE_PERSISTENT).
// pa_reduce_kernel -- Phase 2 of the same page: merges the partials of each
//   (sequence, head) with a log-sum-exp reduce.
//
// Hardware mapping (written for sm_103a, not translated from the pages' Triton):
// * Cache layout [block][kv_head][16 tokens][D]: one (block, kv head) is 16
//   rows of D halves.  A 3-D tensor map views a cache as (64-half column,
//   row, 64-column chunk); each K or V tile of a block arrives as ONE TMA box
//   laid out [chunk][16 rows][128 B] with the 128-byte swizzle, so the
//   ldmatrix reads below hit 8 distinct bank groups (a TMA instruction holds
//   its issuing thread for a fixed time, so one box per tile, not per chunk).
// * Each of the NW warps of a CTA owns NS shared-memory stages (K and V of one
//   block each), an mbarrier per stage, and a private online-softmax state;
//   blocks of the partition are dealt round-robin to the warps.  Several CTA
//   shapes (NW, NS) are compiled; the host picks one per call.  Lane 0
//   issues the copies; every wait is bounded (no spin can hang the GPU).
// * Scores and PV run on the tensor cores as m16n8k16 MMAs in swapped form:
//   S^T[16 tokens x 8 heads] = K[16 x D] . Q^T[D x 8] and
//   O^T[D x 8 heads] += V^T[D x 16] . P^T[16 x 8], so the <= 8 heads of a
//   GQA group sit in the N dimension.  P^T reaches the B-operand layout with
//   movmatrix (an in-register 8x8 transpose), with no shared-memory round trip.
// * Softmax state is kept in the log2 domain (scores pre-multiplied by
//   scale*log2 e and exponentiated with exp2f).  Inside a warp the running
//   max is updated per block and the accumulator rescaled by
//   alpha = 2^(m_old - m_new), with the block probabilities taken relative to
//   the new max; this is the alpha/beta update of the
//   "paged_attention_v2_triton.py" commit page with beta folded into p.
#include "pa_internal.h"

#include <math.h>

#include "pa_decode.h"
#include "pa_device.cuh"
#include "pa_partition_block.cuh"

namespace pa {

__device__ unsigned int g_status;

namespace {

#ifdef PA_TRACE
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
#define PA_TRACE_MARK(slot)                                                                              \
    do {                                                                                                 \
        if (prm.trace && threadIdx.x == 0) {                                                             \
            const size_t cta = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;   \
            prm.trace[cta * 5 + (slot)] = global_ns();                                                   \
        }                                                                                                \
    } while (0)
#else
#define PA_TRACE_MARK(slot) \
    do {                    \
    } while (0)
#endif

}  // namespace

// Single-launch merge of the partials (fused combine), run by every thread of
// a partition CTA after its warps wrote their partial.  The CTA publishes the
// partial (fence), takes a ticket for its (sequence, kv head); the CTA that
// draws the last ticket merges the n partials of the G heads and resets the
// ticket for the next call.  No CTA ever waits for another.
//
// The merge: per head, M = max_p m_p and the weights w_p = l_p 2^(m_p - M) /
// sum_p l_p 2^(m_p - M) (one warp per head, into shared memory); then the
// heads' partial rows arrive in the idle stage area in chunks of partitions,
// each head's rows of a chunk as one bulk copy, and every thread adds
// w_p O_p to its own float4 columns of an accumulator in shared memory, in
// partition order -- the same weighted sum as the reduce kernel's fold up to
// rounding, and the bits do not depend on which CTA finished last.  With
// fewer than eight partitions, or when the weights and one partition per
// chunk do not fit the stage area, the merge reads the partials with plain
// loads instead.
template <int D, int NW, int NS>
__device__ __forceinline__ void fused_combine(const PartitionParams& prm, int b, int kvh, int n, uint8_t* smem,
                                              int* s_last, uint32_t bar) {
    using S = PartitionShape<D, NW, NS>;
    __threadfence();
    __syncthreads();
    unsigned int* tk = prm.tickets + 2 * ((size_t)b * prm.num_kv_heads + kvh);
    if (threadIdx.x == 0) *s_last = atomicAdd(tk, 1u) == (unsigned)(n - 1);
    __syncthreads();
    if (!*s_last) return;
    __threadfence();  // the other partials were published before their tickets
    if (threadIdx.x == 0) atomicExch(tk, 0u);
    const int G = prm.group;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t head0 = (size_t)b * prm.num_heads + (size_t)kvh * G;
    const int wbytes = (G * n * 4 + 15) / 16 * 16;  // the weights
    constexpr int kRowBytes = D * 4;                 // one partition of one head
    const int abytes = G * kRowBytes;                // the accumulator
    const int kmax = (S::kStageArea - wbytes - abytes) / (G * kRowBytes);

    // Staging pays from about eight partitions on (GB300: 8 sequences of up to
    // 8192 tokens at 512-token partitions, 37.3 -> 33.3 us per call; with 1024-
    // token partitions, at most 8 of them, 28.6 -> 29.4).
    if (kmax >= 1 && n >= 8) {
        float* wts = reinterpret_cast<float*>(smem);                  // [G][n]
        float4* acc = reinterpret_cast<float4*>(smem + wbytes);       // [G][D / 4]
        float4* rows = reinterpret_cast<float4*>(smem + wbytes + abytes);  // [G][k][D / 4]
        for (int h = warp; h < G; h += NW) {
            const size_t row = (head0 + h) * prm.max_partitions;
            const float* ml = prm.max_logits + row;
            const float* el = prm.exp_sums + row;
            float M = -INFINITY;
            for (int p = lane; p < n; p += 32) M = fmaxf(M, __ldcg(ml + p));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
            float W = 0.f;
            for (int p = lane; p < n; p += 32) {
                const float w = __ldcg(el + p) * exp2f(__ldcg(ml + p) - M);
                wts[h * n + p] = w;
                W += w;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(kFull, W, off);
            const float inv = 1.f / W;
            for (int p = lane; p < n; p += 32) wts[h * n + p] *= inv;  // this lane's own entries
        }
        for (int t = threadIdx.x; t < G * (D / 4); t += NW * 32) acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (threadIdx.x == 0) {
            mbar_init(bar, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        // the stage area was last read and written by this CTA's threads through
        // the generic proxy; the partials were written by other CTAs the same way
        asm volatile("fence.proxy.async;" ::: "memory");
        __syncthreads();
        bool ok = true;
        uint32_t phase = 0;
        for (int p0 = 0; p0 < n && ok; p0 += kmax, phase ^= 1u) {
            const int k = min(kmax, n - p0);
            if (threadIdx.x == 0) {
                mbar_arrive_expect_tx(bar, (uint32_t)(G * k * kRowBytes));
                for (int h = 0; h < G; ++h)
                    bulk_load(smem_addr(rows) + (uint32_t)(h * k * kRowBytes),
                              prm.tmp_out + ((head0 + h) * prm.max_partitions + p0) * D, (uint32_t)(k * kRowBytes), bar);
            }
            if (!mbar_wait(bar, phase, prm.wait_limit)) {
                // the copies still land in this CTA's shared memory: wait for them
                // once more before leaving; the output is not written
                mbar_wait(bar, phase, kDefaultWaitLimit);
                if (threadIdx.x == 0) atomicOr(&g_status, PA_DEV_TIMEOUT);
                ok = false;
            }
            if (ok) {
                for (int t = threadIdx.x; t < G * (D / 4); t += NW * 32) {
                    const int h = t / (D / 4), c4 = t % (D / 4);
                    float4 a = acc[t];
                    for (int q = 0; q < k; ++q) {
                        const float w = wts[h * n + p0 + q];
                        const float4 v = rows[(h * k + q) * (D / 4) + c4];
                        a.x += w * v.x;
                        a.y += w * v.y;
                        a.z += w * v.z;
                        a.w += w * v.w;
                    }
                    acc[t] = a;
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncthreads();  // the chunk is consumed before the next copy overwrites it
        }
        if (!ok) return;
        for (int t = threadIdx.x; t < G * (D / 4); t += NW * 32) {
            const int h = t / (D / 4), c4 = t % (D / 4);
            const float4 a = acc[t];
            __half2* o = reinterpret_cast<__half2*>(prm.out + (head0 + h) * D + 4 * c4);
            o[0] = __floats2half2_rn(a.x, a.y);
            o[1] = __floats2half2_rn(a.z, a.w);
        }
        return;
    }

    // Plain loads: each thread folds its (head, float4 column) tasks over the
    // partitions in order with the alpha/beta rescale of the reduce kernel,
    // four partitions' loads in flight at a time.
    for (int task = threadIdx.x; task < G * (D / 4); task += NW * 32) {
        const int hh = task / (D / 4), col = task % (D / 4);
        const size_t row = (head0 + hh) * prm.max_partitions;
        const float* ml = prm.max_logits + row;
        const float* el = prm.exp_sums + row;
        const float4* tp = reinterpret_cast<const float4*>(prm.tmp_out + row * D) + col;
        float m = -INFINITY, wsum = 0.f;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        auto fold = [&](float mp, float lp, float4 t) {
            const float mn = fmaxf(m, mp);
            const float alpha = exp2f(m - mn);  // 0 on the first partition (m = -inf)
            const float beta = lp * exp2f(mp - mn);
            wsum = wsum * alpha + beta;
            a.x = a.x * alpha + beta * t.x;
            a.y = a.y * alpha + beta * t.y;
            a.z = a.z * alpha + beta * t.z;
            a.w = a.w * alpha + beta * t.w;
            m = mn;
        };
        int p = 0;
        for (; p + 4 <= n; p += 4) {
            float mp[4], lp[4];
            float4 t[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                mp[u] = __ldcg(ml + p + u);
                lp[u] = __ldcg(el + p + u);
                t[u] = __ldcg(tp + (size_t)(p + u) * (D / 4));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) fold(mp[u], lp[u], t[u]);
        }
        for (; p < n; ++p) fold(__ldcg(ml + p), __ldcg(el + p), __ldcg(tp + (size_t)p * (D / 4)));
        const float inv = 1.f / wsum;
        __half2* o = reinterpret_cast<__half2*>(prm.out + (head0 + hh) * D + 4 * col);
        o[0] = __floats2half2_rn(a.x * inv, a.y * inv);
        o[1] = __floats2half2_rn(a.z * inv, a.w * inv);
    }
}

// Parallel merge after a group barrier (FUSED on a co-resident grid, the
// cooperative form).  The n partition CTAs of a (sequence, kv head) publish
// their partials, count themselves in the group's arrival word and wait --
// a bounded wait -- until all n have; then CTA `slot` merges its own slice
// [slot E / n, (slot + 1) E / n) of the group's E = G * D outputs.  Its loads
// go out in one round: the weights w_p = l_p 2^(m_p - M) / sum_q l_q 2^(m_q - M)
// of the heads the slice touches (one warp per head) and the slice's columns
// of every partial, into the idle stage area; then each thread sums w_p O_p
// over p in partition order for its outputs, so the bits do not depend on
// timing.  Every CTA then counts itself in the departure word; the last one
// resets both words (and re-arms a pooled claim counter), so every call
// leaves them zero.  merge = false (an aborted CTA): arrive and depart only.
// The host uses this form only when the staged slice fits the stage area.
template <int D, int NW, int NS>
__device__ __forceinline__ void fused_barrier_merge(const PartitionParams& prm, int b, int kvh, int slot, int n,
                                                    uint8_t* smem, int* s_flag, bool merge) {
    using S = PartitionShape<D, NW, NS>;
    unsigned int* word = prm.tickets + 2 * ((size_t)b * prm.num_kv_heads + kvh);  // arrivals, departures
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        atomicAdd(word, 1u);
        bool ok = false;
        if (merge) {
            for (unsigned it = 0; it < prm.wait_limit; ++it) {
                unsigned v;
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(word) : "memory");
                if (v >= (unsigned)n) {
                    ok = true;
                    break;
                }
            }
            if (!ok) atomicOr(&g_status, PA_DEV_TIMEOUT);
        }
        *s_flag = ok ? 1 : 0;
    }
    __syncthreads();
    if (*s_flag) {
        __threadfence();
        const int G = prm.group, E = G * D;
        const int e0 = (int)((long long)slot * E / n), e1 = (int)((long long)(slot + 1) * E / n);
        const int es = e1 - e0;
        if (es > 0) {
            const int hA = e0 / D, nh = (e1 - 1) / D - hA + 1;  // the heads the slice touches
            const size_t head0 = (size_t)b * prm.num_heads + (size_t)kvh * G;
            float* wts = reinterpret_cast<float*>(smem);  // [nh][n]
            float* acc = wts + ((nh * n + 3) & ~3);       // [n][es]
            const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
            for (int hh = warp; hh < nh; hh += NW) {
                const size_t row = (head0 + hA + hh) * prm.max_partitions;
                float M = -INFINITY;
                for (int p = lane; p < n; p += 32) M = fmaxf(M, __ldcg(prm.max_logits + row + p));
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
                float W = 0.f;
                for (int p = lane; p < n; p += 32) {
                    const float w = __ldcg(prm.exp_sums + row + p) * exp2f(__ldcg(prm.max_logits + row + p) - M);
                    wts[hh * n + p] = w;
                    W += w;
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(kFull, W, off);
                const float inv = 1.f / W;
                for (int p = lane; p < n; p += 32) wts[hh * n + p] *= inv;
            }
            for (int x = threadIdx.x; x < n * es; x += NW * 32) {
                const int p = x / es, e = e0 + x % es;
                acc[x] = __ldcg(prm.tmp_out + ((head0 + e / D) * prm.max_partitions + p) * D + e % D);
            }
            __syncthreads();
            for (int i = threadIdx.x; i < es; i += NW * 32) {
                const int e = e0 + i, hh = e / D - hA;
                float o = 0.f;
                for (int p = 0; p < n; ++p) o += wts[hh * n + p] * acc[p * es + i];
                prm.out[head0 * D + e] = __float2half_rn(o);
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && atomicAdd(word + 1, 1u) == (unsigned)(n - 1)) {
        // every CTA of the group is past the barrier and done claiming
        atomicExch(word, 0u);
        atomicExch(word + 1, 0u);
        if (prm.claims) prm.claims[(size_t)b * prm.num_kv_heads + kvh] = (unsigned long long)kClaimTag << 32;
    }
}

// Bytes of the idle stage area the parallel merge stages for up to n
// partitions of one group (the host checks that this fits before it picks
// that form).  A slice holds es <= ceil(E / n) outputs and touches nh <=
// es / head_dim + 2 heads, so the weights take nh n <= group + 3 n floats
// (+3 to align the columns) and the columns n es <= E + n floats: a bound
// that grows with n, so it covers every group of a plan.
__host__ __device__ constexpr long long barrier_merge_bytes(int n, int group, int head_dim) {
    return 4ll * ((long long)group + (long long)group * head_dim + 4ll * n + 3);
}

// Pooled == false: CTA p takes the blocks of partition p, dealt round-robin
// to its warps.  Pooled == true: the CTAs of a (sequence, kv head) share the
// sequence's blocks in chunks of kPoolChunk; each warp starts with chunk
// p * NW + w and claims further chunks from a device counter, so a warp on a
// faster SM takes more of them and the CTAs finish together.  Every CTA still
// leaves one partial (its warps' merged state); which chunks a partial covers
// then depends on timing, so its rounding can differ from call to call.
template <int D, int NW, int NS, bool Pooled>
__global__ void __launch_bounds__(NW * 32, 1)
    pa_partition_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                        const PartitionParams prm) {
    using S = PartitionShape<D, NW, NS>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kStageArea);
    float* sm_m = reinterpret_cast<float*>(bars + NW * NS);
    float* sm_l = sm_m + NW * kMaxGroup;
    int* sm_abort = reinterpret_cast<int*>(sm_l + NW * kMaxGroup);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t stage0 = smem_addr(smem) + warp * NS * S::kStageBytes;
    const uint32_t bar0 = smem_addr(bars) + warp * NS * 8;

    // Launched as a programmatic dependent of whatever precedes it on the
    // stream: the CTAs may become resident early.  What reads nothing that
    // grid writes -- the copy barriers and the tensor maps' descriptors --
    // is set up before the wait; nothing else is read before the preceding
    // grid has completed and its writes are visible.
    if (threadIdx.x == 0) {
        *sm_abort = 0;
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_v)) : "memory");
    }
    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8 * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Let the dependent reduce launch its CTAs as soon as SMs free up; it
    // still waits for this grid's completion before touching the partials.
    asm volatile("griddepcontrol.launch_dependents;");
#ifdef PA_TRACE
    if (prm.trace && threadIdx.x == 0) {
        unsigned smid;
        asm volatile("mov.u32 %0, %smid;" : "=r"(smid));
        const size_t cta = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        prm.trace[cta * 5 + 0] = smid;
    }
    PA_TRACE_MARK(1);
#endif

    // p: the partition of the sequence; slot: its partial's index in the
    // workspace (they differ only for the partials of a partition range)
    const int p = blockIdx.x + prm.part_begin, slot = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int G = prm.group, H = prm.num_heads;
    const int blocks_per_part = prm.partition_size / kBlockSize;
    const int blk0 = p * blocks_per_part;
    const int32_t* bt = prm.block_tables + (size_t)b * prm.max_blocks_per_seq + blk0;

    // Block ids of this warp's iterations, 32 at a time: lane k of batch n holds
    // the id of iteration 32n + k (block j = warp + it * NW of the partition).
    // The first batch is read before the sequence length is known, bounded by
    // the block-table row, so the two loads overlap.
    const int jmax = max(0, min(blocks_per_part, prm.max_blocks_per_seq - blk0));
    constexpr int C = pool_chunk(NS);  // blocks per chunk of the pooled form
    int ids_copy;
    if constexpr (Pooled) {
        // lane k < C: block k of the warp's first chunk
        const int j = (p * NW + warp) * C + lane;
        ids_copy = (lane < C && j < prm.max_blocks_per_seq)
                       ? __ldg(prm.block_tables + (size_t)b * prm.max_blocks_per_seq + j)
                       : -1;
    } else {
        ids_copy = (warp + lane * NW) < jmax ? __ldg(bt + warp + lane * NW) : -1;
    }
    const int L = __ldg(prm.seq_lens + b);
    int batch_copy = 0;
    auto block_id = [&](int& ids, int& batch, int it) {
        if ((it >> 5) != batch) {
            batch = it >> 5;
            const int j = warp + ((it & ~31) + lane) * NW;
            ids = j < jmax ? __ldg(bt + j) : -1;
        }
        return __shfl_sync(kFull, ids, it & 31);
    };

    if (L < 0 || L > prm.max_seq_len || L > prm.max_blocks_per_seq * kBlockSize) {
        if (slot == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(&g_status, PA_DEV_BAD_SEQ_LEN);
        return;
    }
    // The empty partial of a partition past the sequence's end (partials of a
    // range only): no tokens, so nothing it holds may weigh in a merge.
    auto write_empty_partial = [&]() {
        const size_t head0 = (size_t)b * H + (size_t)kvh * G;
        for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
            const size_t pi = (head0 + i / D) * prm.max_partitions + slot;
            prm.tmp_out[pi * D + i % D] = 0.f;
            if (i % D == 0) {
                prm.max_logits[pi] = -INFINITY;
                prm.exp_sums[pi] = 0.f;
            }
        }
    };
    if (L == 0) {  // empty sequence: the output is zero
        if (prm.partials_only) {
            write_empty_partial();
        } else if (p == 0) {
            for (int i = threadIdx.x; i < G * D; i += blockDim.x)
                prm.out[((size_t)b * H + kvh * G) * D + i] = __float2half_rn(0.f);
        }
        return;
    }
    const int n_part = (L + prm.partition_size - 1) / prm.partition_size;
    if (p >= n_part) {
        if (prm.partials_only) write_empty_partial();
        return;
    }
    const int nblk = min(blocks_per_part, (L + kBlockSize - 1) / kBlockSize - blk0);

    // Blocks j = warp, warp + NW, ... of the partition belong to this warp.
    const int nmine = warp < nblk ? (nblk - warp + NW - 1) / NW : 0;
    uint32_t valid_bits = 0;  // stage s holds a block with a legal id

    // Stage the K and V of block `phys` (the warp's iteration `it`) into stage it % NS.
    auto stage_block = [&](int it, int phys) {
        const int s = it % NS;
        const uint32_t bar = bar0 + 8 * s;
        const bool ok = phys >= 0 && (long long)phys < prm.num_blocks;
        valid_bits = ok ? (valid_bits | (1u << s)) : (valid_bits & ~(1u << s));
        if (lane == 0) {
            if (ok) {
                mbar_arrive_expect_tx(bar, S::kStageBytes);
                const int row = (phys * prm.num_kv_heads + kvh) * kBlockSize;
                const uint32_t kdst = stage0 + s * S::kStageBytes, vdst = kdst + S::kTileBytes;
                // one box per tile: all D / 64 column chunks of the 16 rows
                tma_load_3d(kdst, &tmap_k, 0, row, 0, bar);
                tma_load_3d(vdst, &tmap_v, 0, row, 0, bar);
            } else {
                atomicOr(&g_status, PA_DEV_BAD_BLOCK_ID);
                mbar_arrive(bar);  // complete the phase so the wait below stays in step
            }
        }
    };
    auto issue = [&](int it) { stage_block(it, block_id(ids_copy, batch_copy, it)); };

    // Pooled: chunk q holds blocks [q C, (q + 1) C) of the sequence.  The
    // nw = n_part * NW warps of the sequence's CTAs take chunks round-robin
    // (warp v: v, v + nw, v + 2 nw, ...) up to chunk 3 nw; then a warp's k-th
    // chunk (k >= 3) is 3 nw + the count its claim returned, or, if the
    // counter was not armed, the round-robin one.  The first three need no
    // counter, so the claims of a whole wave of warps do not queue at start.
    const int nblk_seq = (L + kBlockSize - 1) / kBlockSize;
    const int nchunks = (nblk_seq + C - 1) / C;
    const int nw = n_part * NW;
    unsigned long long* const ctr = Pooled ? prm.claims + (size_t)b * prm.num_kv_heads + kvh : nullptr;
    auto chunk_len = [&](int q) { return q < nchunks ? min(C, nblk_seq - q * C) : 0; };
    auto chunk_ids = [&](int q, int len) {
        return lane < len ? __ldg(prm.block_tables + (size_t)b * prm.max_blocks_per_seq + (size_t)q * C + lane) : -1;
    };
    int q_cur = p * NW + warp, len_cur = 0, issued = 0;
    int q_nxt = 0, len_nxt = 0, ids_nxt = -1;
    if constexpr (Pooled) {
        static_assert(NS <= C, "copies run at most one chunk ahead");
        len_cur = chunk_len(q_cur);
        q_nxt = q_cur + nw;
        len_nxt = chunk_len(q_nxt);
        ids_nxt = chunk_ids(q_nxt, len_nxt);
        for (; issued < NS && issued < len_cur; ++issued) stage_block(issued, __shfl_sync(kFull, ids_copy, issued));
    } else {
        for (int it = 0; it < NS && it < nmine; ++it) issue(it);
    }

    const int g = lane >> 2, c = lane & 3;  // MMA fragment row group / column pair

    // Q^T as the B operand of S^T = K . Q^T: lane holds head g, dims 16ks + 2c (+1) and +8.
    uint32_t qb[S::kSteps][2];
    {
        const int hq = g < G ? g : 0;  // lanes of padding heads load nothing
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(prm.q + ((size_t)b * H + kvh * G + hq) * D);
#pragma unroll
        for (int ks = 0; ks < S::kSteps; ++ks) {
            qb[ks][0] = g < G ? __ldg(qrow + 8 * ks + c) : 0u;
            qb[ks][1] = g < G ? __ldg(qrow + 8 * ks + 4 + c) : 0u;
        }
    }

    float o[S::kSteps][4];
#pragma unroll
    for (int i = 0; i < S::kSteps; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;  // running max (log2 domain) of heads 2c, 2c+1
    float l0 = 0.f, l1 = 0.f;              // this lane's share of the exp sums

    const float sl2 = prm.scale_log2;
    int i = 0;
    bool timed_out = false;
    if constexpr (Pooled) {
        // At the start of chunk k the warp holds chunks k and k + 1 (ids
        // loaded a chunk ago), resolves chunk k + 2 from the claim it made at
        // the start of chunk k - 1, loads its ids and claims again; neither
        // latency stalls the copies, which run NS <= C blocks ahead.
        int mode = 0;  // 0: no claim resolved yet, 1: counter armed, 2: round-robin
        bool claimed = false;
        unsigned long long raw = 0;  // lane 0: counter value returned by the last claim
        int q_nn = 0, len_nn = 0, ids_nn = -1;
        for (;; ++i) {
            const int r = i % C;
            if (r == 0) {
                if (i > 0) {
                    q_cur = q_nxt, len_cur = len_nxt, ids_copy = ids_nxt;
                    q_nxt = q_nn, len_nxt = len_nn, ids_nxt = ids_nn;
                }
                if (len_cur == 0) break;
                if (i == 0 || mode == 2) {
                    q_nn = q_nxt + nw;
                } else if (claimed) {
                    const unsigned long long got = __shfl_sync(kFull, raw, 0);
                    if (mode == 0) mode = (unsigned)(got >> 32) == kClaimTag ? 1 : 2;
                    const unsigned cnt = (unsigned)got;  // claims before this one
                    q_nn = mode == 2 ? q_nxt + nw : cnt < (unsigned)nchunks ? 3 * nw + (int)cnt : nchunks;
                } else {
                    q_nn = nchunks;  // the previous chunk resolved was past the end
                }
                len_nn = chunk_len(q_nn);
                ids_nn = chunk_ids(q_nn, len_nn);
                claimed = mode != 2 && len_nn > 0;
                if (claimed && lane == 0) raw = atomicAdd(ctr, 1ull);
            }
            if (r >= len_cur) break;
            const int s = i % NS;
            const uint32_t bar = bar0 + 8 * s;
            if (prm.force_timeout || !mbar_wait(bar, (i / NS) & 1, prm.wait_limit)) {
                timed_out = true;
                break;
            }
            if (i == 0) PA_TRACE_MARK(2);
            if ((valid_bits >> s) & 1u) {
                const int tok0 = (q_cur * C + r) * kBlockSize;
                const uint32_t kst = stage0 + s * S::kStageBytes;
                warp_block_update<D>(qb, o, m0, m1, l0, l1, kst, kst + S::kTileBytes,
                                     smem + (kst + S::kTileBytes - smem_addr(smem)), min(kBlockSize, L - tok0),
                                     sl2);
            }
            __syncwarp();
            const int rn = r + NS;  // chunk-relative block of iteration i + NS
            if (rn < C) {
                if (rn < len_cur) stage_block(issued++, __shfl_sync(kFull, ids_copy, rn));
            } else if (rn - C < len_nxt) {
                stage_block(issued++, __shfl_sync(kFull, ids_nxt, rn - C));
            }
        }
    } else {
    for (; i < nmine; ++i) {
        const int s = i % NS;
        const uint32_t bar = bar0 + 8 * s;
        if (prm.force_timeout || !mbar_wait(bar, (i / NS) & 1, prm.wait_limit)) {
            timed_out = true;
            break;
        }
        if (i == 0) PA_TRACE_MARK(2);
        if ((valid_bits >> s) & 1u) {
            const int tok0 = (blk0 + warp + i * NW) * kBlockSize;
            const uint32_t kst = stage0 + s * S::kStageBytes;
            warp_block_update<D>(qb, o, m0, m1, l0, l1, kst, kst + S::kTileBytes,
                                 smem + (kst + S::kTileBytes - smem_addr(smem)), min(kBlockSize, L - tok0), sl2);
        }
        __syncwarp();
        if (i + NS < nmine) issue(i + NS);
    }
    issued = min(nmine, i + NS);
    }

    if (timed_out) {
        // Drain this warp's copies still in flight before the CTA may exit.
        for (int k = i; k < issued; ++k) mbar_wait(bar0 + 8 * (k % NS), (k / NS) & 1, kDefaultWaitLimit);
        if (lane == 0) {
            atomicOr(&g_status, PA_DEV_TIMEOUT);
            atomicExch(sm_abort, 1);
        }
    }

    // Finish this warp's exp sums: add the shares of the 8 lanes holding the same heads.
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(kFull, l0, off);
        l1 += __shfl_xor_sync(kFull, l1, off);
    }
    __syncthreads();  // all stages consumed; the stage area is reused below
    PA_TRACE_MARK(3);
    if (*sm_abort) {
        // A fused combine counts every partition's ticket, so an aborted CTA
        // still takes its own; the last one resets the count (the output is
        // not written and the status word already reports the failure).
        if (prm.tickets && n_part > 1) {
            if (prm.coop) {
                fused_barrier_merge<D, NW, NS>(prm, b, kvh, slot, n_part, smem, sm_abort + 1, false);
            } else if (threadIdx.x == 0) {
                unsigned int* tk = prm.tickets + 2 * ((size_t)b * prm.num_kv_heads + kvh);
                if (atomicAdd(tk, 1u) == (unsigned)(n_part - 1)) atomicExch(tk, 0u);
            }
        }
        return;
    }

    const bool fused = prm.tickets && n_part > 1;
    const bool direct = n_part == 1 && !prm.partials_only;
    if constexpr (NW == 1) {
    // One warp: the output is its own state, o / l, stored from the MMA
    // fragments (lane (g, c) holds heads 2c, 2c + 1).  A partition whose
    // blocks all had illegal ids (m = -inf) was reported above.
    const float w0 = m0 == -INFINITY ? 0.f : 1.f, w1 = m1 == -INFINITY ? 0.f : 1.f;
    const float L0 = w0 * l0, L1 = w1 * l1;
    const float f0 = w0 * (1.f / L0), f1 = w1 * (1.f / L1);
    const bool has0 = 2 * c < G, has1 = 2 * c + 1 < G;  // padding heads are not written
    const size_t head0 = (size_t)b * H + kvh * G + 2 * c;
    const size_t pi0 = head0 * prm.max_partitions + slot, pi1 = pi0 + prm.max_partitions;
#pragma unroll
    for (int mt = 0; mt < S::kSteps; ++mt) {
        const int d = 16 * mt + g;
        const float v00 = f0 * o[mt][0], v10 = f1 * o[mt][1];  // (head 2c, d), (head 2c+1, d)
        const float v08 = f0 * o[mt][2], v18 = f1 * o[mt][3];  // ... at d + 8
        if (direct) {
            if (has0) {
                prm.out[head0 * D + d] = __float2half_rn(v00);
                prm.out[head0 * D + d + 8] = __float2half_rn(v08);
            }
            if (has1) {
                prm.out[(head0 + 1) * D + d] = __float2half_rn(v10);
                prm.out[(head0 + 1) * D + d + 8] = __float2half_rn(v18);
            }
        } else {
            if (has0) {
                prm.tmp_out[pi0 * D + d] = v00;
                prm.tmp_out[pi0 * D + d + 8] = v08;
            }
            if (has1) {
                prm.tmp_out[pi1 * D + d] = v10;
                prm.tmp_out[pi1 * D + d + 8] = v18;
            }
        }
    }
    if (!direct && g == 0) {
        if (has0) {
            prm.max_logits[pi0] = m0;
            prm.exp_sums[pi0] = L0;
        }
        if (has1) {
            prm.max_logits[pi1] = m1;
            prm.exp_sums[pi1] = L1;
        }
    }
    } else {
    // Merge the NW partial states of this CTA by the same max/rescale rule.
    // Every warp leaves (m, l, O) in shared memory; then warp w merges dims
    // [w D/NW, (w+1) D/NW) of every head: lane (h, q) = (lane / 4, lane % 4)
    // takes head h and the dim pairs 2q, 2q + 1 of each 8-dim group, so a
    // head's stores are contiguous.  The sums run in warp order, as in the
    // one-warp form, so the bits do not depend on which warp merges.
    float* red = reinterpret_cast<float*>(smem);  // [NW][kMaxGroup][kRedStride]
    {
        float* rw = red + warp * kMaxGroup * S::kRedStride;
#pragma unroll
        for (int mt = 0; mt < S::kSteps; ++mt) {
            const int d = 16 * mt + g;
            rw[(2 * c) * S::kRedStride + d] = o[mt][0];
            rw[(2 * c + 1) * S::kRedStride + d] = o[mt][1];
            rw[(2 * c) * S::kRedStride + d + 8] = o[mt][2];
            rw[(2 * c + 1) * S::kRedStride + d + 8] = o[mt][3];
        }
        if (g == 0) {
            sm_m[warp * kMaxGroup + 2 * c] = m0;
            sm_m[warp * kMaxGroup + 2 * c + 1] = m1;
            sm_l[warp * kMaxGroup + 2 * c] = l0;
            sm_l[warp * kMaxGroup + 2 * c + 1] = l1;
        }
    }
    __syncthreads();
    constexpr int kSlice = D / NW;  // dims merged by one warp
    static_assert(kSlice % 8 == 0, "a warp merges whole 8-dim groups");
    const int h = lane >> 2, qd = lane & 3;
    if (h < G) {  // padding heads are not written
        // M = max over warps, f_w = 2^(m_w - M) / L, L = sum_w 2^(m_w - M) l_w
        // (warps without blocks have m_w = -inf and contribute nothing)
        float Mh = sm_m[h];
#pragma unroll
        for (int w = 1; w < NW; ++w) Mh = fmaxf(Mh, sm_m[w * kMaxGroup + h]);
        float f[NW];
        f[0] = sm_m[h] == -INFINITY ? 0.f : exp2f(sm_m[h] - Mh);
        float Lh = f[0] * sm_l[h];
#pragma unroll
        for (int w = 1; w < NW; ++w) {
            const float mw = sm_m[w * kMaxGroup + h];
            f[w] = mw == -INFINITY ? 0.f : exp2f(mw - Mh);
            Lh += f[w] * sm_l[w * kMaxGroup + h];
        }
        const float inv = 1.f / Lh;
#pragma unroll
        for (int w = 0; w < NW; ++w) f[w] *= inv;
        const size_t head = (size_t)b * H + kvh * G + h;
        const size_t pi = head * prm.max_partitions + slot;
#pragma unroll
        for (int k = 0; k < kSlice / 8; ++k) {
            const int d = warp * kSlice + 8 * k + 2 * qd;
            const float* r0 = red + h * S::kRedStride + d;
            float v0 = f[0] * r0[0], v1 = f[0] * r0[1];
#pragma unroll
            for (int w = 1; w < NW; ++w) {
                const float* rw = red + (w * kMaxGroup + h) * S::kRedStride + d;
                v0 += f[w] * rw[0];
                v1 += f[w] * rw[1];
            }
            if (direct)
                *reinterpret_cast<__half2*>(prm.out + head * D + d) = __floats2half2_rn(v0, v1);
            else
                *reinterpret_cast<float2*>(prm.tmp_out + pi * D + d) = make_float2(v0, v1);
        }
        if (!direct && warp == 0 && qd == 0) {
            prm.max_logits[pi] = Mh;
            prm.exp_sums[pi] = Lh;
        }
    }
    }
    // spare words of the control area: the ticket result, then an 8-byte copy barrier
    if (fused) {
        if (prm.coop)
            fused_barrier_merge<D, NW, NS>(prm, b, kvh, slot, n_part, smem, sm_abort + 1, true);
        else
            fused_combine<D, NW, NS>(prm, b, kvh, n_part, smem, sm_abort + 1, smem_addr(sm_abort + 2));
    }
    PA_TRACE_MARK(4);
}

// Phase 2: merge the partials of each (sequence, head).  With M = max_p m_p,
// out = sum_p w_p acc_p / sum_p w_p and w_p = l_p 2^(m_p - M): the
// log-sum-exp merge.  One CTA per (head, sequence, W-wide slice of head_dim);
// W/4 threads cover the slice with float4 loads and the remaining factor of
// the 256 threads strides over the partitions.  Each thread folds its
// partitions in order with the alpha/beta rescale of the
// "paged_attention_v2_triton.py" commit page (running max m, alpha =
// 2^(m_old - m_new), beta = l_p 2^(m_p - m_new)), so no separate pass for
// the max is needed; the groups are then merged by the same rule in a fixed
// order, which keeps results deterministic.
// Merge: the partials were gathered from several sources (split-KV across
// devices; see ReduceParams::src_parts), and every sequence's output is
// written here, also for one partition or none.
template <int D, int W, bool Merge>
__global__ void __launch_bounds__(kReduceThreads) pa_reduce_kernel(const ReduceParams prm) {
    constexpr int kLanes = W / 4;                    // float4 columns of a slice
    constexpr int kGroups = kReduceThreads / kLanes; // partition groups
    static_assert(W <= D && D % W == 0 && kLanes <= kReduceThreads, "slice width");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int h = blockIdx.x, b = blockIdx.y, slice = blockIdx.z;
    // re-arm the pooled split's claim counter of (b, kv head h / group): the
    // partition grid that used it has completed
    if (prm.claims && slice == 0 && h % prm.group == 0 && threadIdx.x == 0)
        prm.claims[(size_t)b * (prm.num_heads / prm.group) + h / prm.group] = (unsigned long long)kClaimTag << 32;
    const size_t base = ((size_t)b * prm.num_heads + h) * (Merge ? prm.src_parts : prm.max_partitions);
    const float* ml = prm.max_logits + base;
    const float* el = prm.exp_sums + base;
    const int col = threadIdx.x % kLanes, pg = threadIdx.x / kLanes;
    const float4* tp = reinterpret_cast<const float4*>(prm.tmp_out + base * D + slice * W) + col;
    // offset of partition p from base: slot p % src_parts of source p / src_parts
    auto at = [&](int p) -> size_t {
        if constexpr (Merge) {
            const int r = p / prm.src_parts;
            return (size_t)r * prm.src_stride + (size_t)(p - r * prm.src_parts);
        } else {
            return (size_t)p;
        }
    };
    // A thread's first kPre partials are read together with the length, so
    // their latencies overlap: the row holds max_partitions entries, so the
    // reads stay inside the workspace, and a value past the sequence's
    // partitions is never used.
    constexpr int kPre = 2;
    float mp0[kPre], lp0[kPre];
    float4 t0[kPre];
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
        const int p = pg + i * kGroups;
        mp0[i] = lp0[i] = 0.f;
        t0[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p < prm.max_partitions) {
            mp0[i] = ml[at(p)];
            lp0[i] = el[at(p)];
            t0[i] = tp[at(p) * (D / 4)];
        }
    }
    const int L = prm.seq_lens[b];
    const int part = prm.part_sizes ? prm.part_sizes[b] : prm.partition_size;
    if constexpr (Merge) {
        if (L < 0 || L > prm.max_seq_len || L > prm.max_blocks_per_seq * kBlockSize) {
            if (h == 0 && slice == 0 && threadIdx.x == 0) atomicOr(&g_status, PA_DEV_BAD_SEQ_LEN);
            return;
        }
        if (L == 0) {  // empty sequence: the output is zero
            if (threadIdx.x < W)
                prm.out[((size_t)b * prm.num_heads + h) * D + slice * W + threadIdx.x] = __float2half_rn(0.f);
            return;
        }
    } else if (L <= 0 || L > prm.max_seq_len || L > prm.max_blocks_per_seq * kBlockSize) {
        // single-partition, empty and invalid sequences were finished by the partition kernel
        return;
    }
    // (a flat split's count comes from the workspace: clamped to the row, so a
    // stale word could never send the reads past it)
    const int n = prm.part_counts ? min(prm.part_counts[b], prm.max_partitions) : (L + part - 1) / part;
    if (!Merge && n <= 1) return;

    __shared__ float4 red_acc[kGroups][kLanes];
    __shared__ float red_m[kGroups];
    __shared__ float red_w[kGroups];

    float m = -INFINITY, wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto fold = [&](float mp, float lp, const float4& t) {
        const float mn = fmaxf(m, mp);
        const float alpha = exp2f(m - mn);  // 0 on the first partition (m = -inf)
        const float beta = lp * exp2f(mp - mn);
        wsum = wsum * alpha + beta;
        acc.x = acc.x * alpha + beta * t.x;
        acc.y = acc.y * alpha + beta * t.y;
        acc.z = acc.z * alpha + beta * t.z;
        acc.w = acc.w * alpha + beta * t.w;
        m = mn;
    };
#pragma unroll
    for (int i = 0; i < kPre; ++i)
        if (pg + i * kGroups < n) fold(mp0[i], lp0[i], t0[i]);
#pragma unroll 4
    for (int p = pg + kPre * kGroups; p < n; p += kGroups) fold(ml[at(p)], el[at(p)], tp[at(p) * (D / 4)]);
    red_acc[pg][col] = acc;
    if (col == 0) {
        red_m[pg] = m;
        red_w[pg] = wsum;
    }
    __syncthreads();
    if (threadIdx.x < W) {
        const int dl = threadIdx.x;
        float M = -INFINITY;
#pragma unroll 8
        for (int q = 0; q < kGroups; ++q) M = fmaxf(M, red_m[q]);
        float sum = 0.f, wt = 0.f;
#pragma unroll 8
        for (int q = 0; q < kGroups; ++q) {
            const float f = red_m[q] == -INFINITY ? 0.f : exp2f(red_m[q] - M);  // groups without partitions
            sum += f * reinterpret_cast<const float*>(red_acc[q])[dl];
            wt += f * red_w[q];
        }
        prm.out[((size_t)b * prm.num_heads + h) * D + slice * W + dl] = __float2half_rn(sum / wt);
    }
}

// The CTA shapes (warps, stages per warp) compiled for every head_dim.
#define PA_FOR_EACH_SHAPE(X) X(2, 2) X(1, 2) X(1, 3) X(4, 2)

int partition_smem_bytes(int head_dim, int warps, int stages) {
#define PA_SMEM_CASE(W_, S_)                                                       \
    if (warps == W_ && stages == S_) {                                            \
        switch (head_dim) {                                                       \
            case 64: return PartitionShape<64, W_, S_>::kSmemBytes;               \
            case 128: return PartitionShape<128, W_, S_>::kSmemBytes;             \
            case 256: return PartitionShape<256, W_, S_>::kSmemBytes;             \
            default: return -1;                                                   \
        }                                                                         \
    }
    PA_FOR_EACH_SHAPE(PA_SMEM_CASE)
#undef PA_SMEM_CASE
    return -1;
}

namespace {

template <int D, int NW, int NS, bool Pooled>
cudaError_t launch_partition_t(const PartitionParams& prm, const CUtensorMap& tk, const CUtensorMap& tv, dim3 grid,
                               cudaStream_t stream) {
    const int smem = PartitionShape<D, NW, NS>::kSmemBytes;
    static std::atomic<unsigned long long> done{0};
    static int resident[64];  // CTAs one SM holds at once, per device (for the cooperative form)
    cudaError_t e = once_per_device(done, [&] {
        cudaError_t r = cudaFuncSetAttribute(pa_partition_kernel<D, NW, NS, Pooled>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (r != cudaSuccess) return r;
        // all of an SM's shared memory, so that the dependent reduce CTAs fit beside these
        r = cudaFuncSetAttribute(pa_partition_kernel<D, NW, NS, Pooled>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
        if (r != cudaSuccess) return r;
        int dev = 0, per_sm = 0, sms = 0;
        if ((r = cudaGetDevice(&dev)) != cudaSuccess) return r;
        if ((r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pa_partition_kernel<D, NW, NS, Pooled>,
                                                               NW * 32, smem)) != cudaSuccess)
            return r;
        if ((r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return r;
        if (dev >= 0 && dev < 64) resident[dev] = per_sm * sms;
        return cudaSuccess;
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2] = {pdl_attribute(), {}};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (prm.coop) {
        // every CTA resident at once, or no launch at all: the CTAs of a group wait for each other
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        const long long ctas = (long long)grid.x * grid.y * grid.z;
        if (dev < 0 || dev >= 64 || ctas > resident[dev]) return cudaErrorCooperativeLaunchTooLarge;
        attr[1].id = cudaLaunchAttributeCooperative;
        attr[1].val.cooperative = 1;
        cfg.numAttrs = 2;
    }
    e = cudaLaunchKernelEx(&cfg, pa_partition_kernel<D, NW, NS, Pooled>, tk, tv, prm);
    if (e != cudaSuccess && prm.coop) {
        // a cooperative launch that the runtime will not combine with the
        // programmatic dependency: launch it as a plain stream successor
        cudaGetLastError();
        attr[0] = attr[1];
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, pa_partition_kernel<D, NW, NS, Pooled>, tk, tv, prm);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D, int W, bool Merge>
cudaError_t launch_reduce_t(const ReduceParams& prm, dim3 grid, cudaStream_t stream) {
    // The largest shared-memory carveout, as the partition kernel's needs: an
    // SM runs CTAs of one carveout at a time, so with a smaller one the
    // reduce CTAs could not become resident beside the partition CTAs that
    // they wait on.
    static std::atomic<unsigned long long> done{0};
    cudaError_t e = once_per_device(done, [] {
        return cudaFuncSetAttribute(pa_reduce_kernel<D, W, Merge>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    (int)cudaSharedmemCarveoutMaxShared);
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kReduceThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, pa_reduce_kernel<D, W, Merge>, prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D, bool Merge>
cudaError_t launch_reduce_m(int width, const ReduceParams& prm, dim3 grid, cudaStream_t stream) {
    switch (width) {
        case 32: return launch_reduce_t<D, 32, Merge>(prm, grid, stream);
        case 64: return launch_reduce_t<D, 64, Merge>(prm, grid, stream);
        case 128: if constexpr (D >= 128) return launch_reduce_t<D, 128, Merge>(prm, grid, stream); else break;
        case 256: if constexpr (D >= 256) return launch_reduce_t<D, 256, Merge>(prm, grid, stream); else break;
        default: break;
    }
    return cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_reduce_d(int width, const ReduceParams& prm, dim3 grid, cudaStream_t stream) {
    return prm.src_parts > 0 ? launch_reduce_m<D, true>(width, prm, grid, stream)
                             : launch_reduce_m<D, false>(width, prm, grid, stream);
}

}  // namespace

cudaError_t launch_partition(int head_dim, int warps, int stages, const PartitionParams& prm, const CUtensorMap& tk,
                             const CUtensorMap& tv, dim3 grid, cudaStream_t stream) {
#define PA_LAUNCH_CASE(W_, S_)                                                                     \
    if (warps == W_ && stages == S_) {                                                            \
        const bool pooled = prm.claims != nullptr;                                                \
        switch (head_dim) {                                                                       \
            case 64:                                                                              \
                return pooled ? launch_partition_t<64, W_, S_, true>(prm, tk, tv, grid, stream)   \
                              : launch_partition_t<64, W_, S_, false>(prm, tk, tv, grid, stream); \
            case 128:                                                                             \
                return pooled ? launch_partition_t<128, W_, S_, true>(prm, tk, tv, grid, stream)  \
                              : launch_partition_t<128, W_, S_, false>(prm, tk, tv, grid, stream); \
            case 256:                                                                             \
                return pooled ? launch_partition_t<256, W_, S_, true>(prm, tk, tv, grid, stream)  \
                              : launch_partition_t<256, W_, S_, false>(prm, tk, tv, grid, stream); \
            default: return cudaErrorInvalidValue;                                                \
        }                                                                                         \
    }
    PA_FOR_EACH_SHAPE(PA_LAUNCH_CASE)
#undef PA_LAUNCH_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_reduce(int head_dim, int width, const ReduceParams& prm, dim3 grid, cudaStream_t stream) {
    switch (head_dim) {
        case 64: return launch_reduce_d<64>(width, prm, grid, stream);
        case 128: return launch_reduce_d<128>(width, prm, grid, stream);
        case 256: return launch_reduce_d<256>(width, prm, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

long long fused_barrier_bytes(int n, int group, int head_dim) { return barrier_merge_bytes(n, group, head_dim); }

cudaError_t disarm_claims(unsigned long long* claims, size_t count, cudaStream_t stream) {
    return cudaMemsetAsync(claims, 0, count * sizeof(unsigned long long), stream);
}

unsigned int* device_status_ptr() {
    constexpr int kMaxDev = 64;
    static unsigned int* cached[kMaxDev];  // a symbol's address is fixed for the context's lifetime
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    if (dev >= 0 && dev < kMaxDev && cached[dev]) return cached[dev];
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    if (dev >= 0 && dev < kMaxDev) cached[dev] = static_cast<unsigned int*>(p);
    return static_cast<unsigned int*>(p);
}

cudaError_t read_and_clear_status(cudaStream_t stream, int* status) {
    unsigned int v = 0;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
    *status = static_cast<int>(v);
    return cudaSuccess;
}

}  // namespace pa
