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
// a partition CTA after warp 0 wrote its partial.  The CTA publishes the
// partial (fence), takes a ticket for its (sequence, kv head); the CTA that
// draws the last ticket merges the n partials of the G heads in partition
// order -- the log-sum-exp fold of the reduce kernel, so the result does not
// depend on which CTA finished last -- and resets the ticket for the next
// call.  No CTA ever waits for another.  Four partitions' loads are in
// flight per thread at a time.
template <int D, int NW>
__device__ __forceinline__ void fused_combine(const PartitionParams& prm, int b, int kvh, int n, int* s_last) {
    __threadfence();
    __syncthreads();
    unsigned int* tk = prm.tickets + (size_t)b * prm.num_kv_heads + kvh;
    if (threadIdx.x == 0) *s_last = atomicAdd(tk, 1u) == (unsigned)(n - 1);
    __syncthreads();
    if (!*s_last) return;
    __threadfence();  // the other partials were published before their tickets
    if (threadIdx.x == 0) atomicExch(tk, 0u);
    const int G = prm.group;
    const size_t head0 = (size_t)b * prm.num_heads + (size_t)kvh * G;
    for (int task = threadIdx.x; task < G * (D / 4); task += NW * 32) {
        const int hh = task / (D / 4), col = task % (D / 4);
        const size_t row = (head0 + hh) * prm.max_partitions;
        const float* ml = prm.max_logits + row;
        const float* el = prm.exp_sums + row;
        const float4* tp = reinterpret_cast<const float4*>(prm.tmp_out + row * D) + col;
        float m = -INFINITY, wsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        auto fold = [&](float mp, float lp, float4 t) {
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
        o[0] = __floats2half2_rn(acc.x * inv, acc.y * inv);
        o[1] = __floats2half2_rn(acc.z * inv, acc.w * inv);
    }
}

template <int D, int NW, int NS>
struct PartitionShape {
    static constexpr int kSteps = D / 16;                      // k-steps of QK, m-tiles of PV
    static constexpr int kChunks = D / 64;                     // TMA boxes per K (or V) block
    static constexpr int kBoxBytes = kBlockSize * 128;         // 16 rows x 64 halves
    static constexpr int kTileBytes = kBlockSize * D * 2;      // K (or V) of one block
    static constexpr int kStageBytes = 2 * kTileBytes;         // K + V
    static constexpr int kStageArea = NW * NS * kStageBytes;
    static constexpr int kRedStride = D + 4;                   // padded row of the cross-warp reduce
    static constexpr int kRedBytes = NW * kMaxGroup * kRedStride * 4;
    static constexpr int kCtrlBytes = NW * NS * 8 + 2 * NW * kMaxGroup * 4 + 16;
    static constexpr int kSmemBytes = 1024 + kStageArea + kCtrlBytes;
    static_assert(kRedBytes <= kStageArea, "cross-warp reduce must fit in the stage area");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget of one CTA");
};

// One 16-token block of a warp's online softmax, in the swapped MMA form:
// S^T = K . Q^T, the running-max update with rescale alpha = 2^(m_old - m_new),
// P^T by movmatrix, then O^T += V^T . P^T.  `kst`/`vst` are the block's K and
// V stages (shared-memory addresses, 64-column boxes with the 128-byte
// swizzle), `vgen` the V stage as a generic pointer: rows from `nvalid` on are
// cleared there before P.V reads them.  Lane (g, c) holds heads 2c, 2c + 1.
template <int D>
__device__ __forceinline__ void warp_block_update(const uint32_t (&qb)[D / 16][2], float (&o)[D / 16][4], float& m0,
                                                  float& m1, float& l0, float& l1, uint32_t kst, uint32_t vst,
                                                  uint8_t* vgen, int nvalid, float sl2) {
    constexpr int kSteps = D / 16, kChunks = D / 64, kBoxBytes = kBlockSize * 128;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int mi = lane >> 3, r8 = lane & 7;
    const int rq = r8 + ((mi & 1) << 3);   // ldmatrix row (token) for K . Q^T
    const int rv = r8 + ((mi >> 1) << 3);  // ldmatrix row (token) for V^T . P^T

    // S^T = K . Q^T  (two accumulators for instruction-level parallelism)
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < kSteps; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, kst + (ks >> 2) * kBoxBytes + swz(rq, ((ks & 3) << 1) + (mi >> 1)));
        if (ks & 1)
            mma_16816(sb, a, qb[ks][0], qb[ks][1]);
        else
            mma_16816(sa, a, qb[ks][0], qb[ks][1]);
    }
    // lane holds tokens g (s0, s1) and g + 8 (s2, s3) of heads 2c, 2c + 1
    float s0 = (sa[0] + sb[0]) * sl2, s1 = (sa[1] + sb[1]) * sl2;
    float s2 = (sa[2] + sb[2]) * sl2, s3 = (sa[3] + sb[3]) * sl2;
    if (g >= nvalid) s0 = s1 = -INFINITY;  // tokens past the end are excluded
    if (g + 8 >= nvalid) s2 = s3 = -INFINITY;

    float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, off));
        bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, off));
    }
    const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    const __half2 p01 = __floats2half2_rn(exp2f(s0 - mn0), exp2f(s1 - mn1));
    const __half2 p23 = __floats2half2_rn(exp2f(s2 - mn0), exp2f(s3 - mn1));
    // the exp sums use the rounded probabilities that enter P.V
    const float2 f01 = __half22float2(p01), f23 = __half22float2(p23);
    l0 = l0 * al0 + (f01.x + f23.x);
    l1 = l1 * al1 + (f01.y + f23.y);
    if (__any_sync(kFull, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int mt = 0; mt < kSteps; ++mt) {
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
        }
    }
    const uint32_t pb0 = movmatrix_trans(half2_bits(p01));  // P^T rows: heads; cols: tokens 0..7
    const uint32_t pb1 = movmatrix_trans(half2_bits(p23));  // tokens 8..15

    if (nvalid < kBlockSize) {
        // Slots past the end may hold anything (even NaN); 0 * NaN would
        // poison P.V, so clear those V rows before the MMA reads them.
        const int units = (kBlockSize - nvalid) * kChunks * 8;
        for (int u = lane; u < units; u += 32) {
            const int r = nvalid + u / (kChunks * 8), rem = u % (kChunks * 8);
            *reinterpret_cast<uint4*>(vgen + (rem >> 3) * kBoxBytes + r * 128 + (rem & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
    }

    // O^T += V^T . P^T
#pragma unroll
    for (int mt = 0; mt < kSteps; ++mt) {
        uint32_t a[4];
        ldsm_x4_trans(a, vst + (mt >> 2) * kBoxBytes + swz(rv, ((mt & 3) << 1) + (mi & 1)));
        mma_16816(o[mt], a, pb0, pb1);
    }
}

template <int D, int NW, int NS>
__global__ void __launch_bounds__(NW * 32, 1)
    pa_partition_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                        const PartitionParams prm) {
    using S = PartitionShape<D, NW, NS>;
    // Launched as a programmatic dependent of whatever precedes it on the
    // stream: the CTAs may become resident early, but nothing is read before
    // the preceding grid has completed and its writes are visible.
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

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kStageArea);
    float* sm_m = reinterpret_cast<float*>(bars + NW * NS);
    float* sm_l = sm_m + NW * kMaxGroup;
    int* sm_abort = reinterpret_cast<int*>(sm_l + NW * kMaxGroup);

    const int p = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = prm.group, H = prm.num_heads;
    const int blocks_per_part = prm.partition_size / kBlockSize;
    const int blk0 = p * blocks_per_part;
    const int32_t* bt = prm.block_tables + (size_t)b * prm.max_blocks_per_seq + blk0;

    // Block ids of this warp's iterations, 32 at a time: lane k of batch n holds
    // the id of iteration 32n + k (block j = warp + it * NW of the partition).
    // The first batch is read before the sequence length is known, bounded by
    // the block-table row, so the two loads overlap.
    const int jmax = max(0, min(blocks_per_part, prm.max_blocks_per_seq - blk0));
    int ids_copy = (warp + lane * NW) < jmax ? __ldg(bt + warp + lane * NW) : -1;
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
        if (p == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(&g_status, PA_DEV_BAD_SEQ_LEN);
        return;
    }
    if (L == 0) {  // empty sequence: the output is zero
        if (p == 0)
            for (int i = threadIdx.x; i < G * D; i += blockDim.x)
                prm.out[((size_t)b * H + kvh * G) * D + i] = __float2half_rn(0.f);
        return;
    }
    const int n_part = (L + prm.partition_size - 1) / prm.partition_size;
    if (p >= n_part) return;
    const int nblk = min(blocks_per_part, (L + kBlockSize - 1) / kBlockSize - blk0);

    const uint32_t stage0 = smem_addr(smem) + warp * NS * S::kStageBytes;
    const uint32_t bar0 = smem_addr(bars) + warp * NS * 8;
    if (threadIdx.x == 0) *sm_abort = 0;
    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8 * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // Blocks j = warp, warp + NW, ... of the partition belong to this warp.
    const int nmine = warp < nblk ? (nblk - warp + NW - 1) / NW : 0;
    uint32_t valid_bits = 0;  // stage s holds a block with a legal id

    // Stage the K and V of iteration `it` into stage it % NS.
    auto issue = [&](int it) {
        const int phys = block_id(ids_copy, batch_copy, it);
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
    for (int it = 0; it < NS && it < nmine; ++it) issue(it);

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

    if (timed_out) {
        // Drain this warp's copies still in flight before the CTA may exit.
        for (int k = i; k < nmine && k < i + NS; ++k)
            mbar_wait(bar0 + 8 * (k % NS), (k / NS) & 1, kDefaultWaitLimit);
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
        if (prm.tickets && n_part > 1 && threadIdx.x == 0) {
            unsigned int* tk = prm.tickets + (size_t)b * prm.num_kv_heads + kvh;
            if (atomicAdd(tk, 1u) == (unsigned)(n_part - 1)) atomicExch(tk, 0u);
        }
        return;
    }

    // Merge the NW partial states of this CTA by the same max/rescale
    // rule: warps 1.. leave theirs in shared memory, warp 0 folds them into its
    // own MMA fragments with per-head factors and stores straight from registers.
    float* red = reinterpret_cast<float*>(smem);  // [NW - 1][kMaxGroup][kRedStride]
    if (warp > 0) {
        float* rw = red + (warp - 1) * kMaxGroup * S::kRedStride;
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
    const bool fused = prm.tickets && n_part > 1;
    if (warp != 0 && !fused) return;
    if (warp == 0) {
    // Per-head factors for heads 2c and 2c + 1: M = max over warps,
    // f_w = 2^(m_w - M) / L with L = sum_w 2^(m_w - M) l_w (warps without
    // blocks have m_w = -inf and contribute nothing).
    float M0 = m0, M1 = m1;
#pragma unroll
    for (int w = 1; w < NW; ++w) {
        M0 = fmaxf(M0, sm_m[w * kMaxGroup + 2 * c]);
        M1 = fmaxf(M1, sm_m[w * kMaxGroup + 2 * c + 1]);
    }
    float f0[NW], f1[NW];
    f0[0] = m0 == -INFINITY ? 0.f : exp2f(m0 - M0);
    f1[0] = m1 == -INFINITY ? 0.f : exp2f(m1 - M1);
    float L0 = f0[0] * l0, L1 = f1[0] * l1;
#pragma unroll
    for (int w = 1; w < NW; ++w) {
        const float mw0 = sm_m[w * kMaxGroup + 2 * c], mw1 = sm_m[w * kMaxGroup + 2 * c + 1];
        f0[w] = mw0 == -INFINITY ? 0.f : exp2f(mw0 - M0);
        f1[w] = mw1 == -INFINITY ? 0.f : exp2f(mw1 - M1);
        L0 += f0[w] * sm_l[w * kMaxGroup + 2 * c];
        L1 += f1[w] * sm_l[w * kMaxGroup + 2 * c + 1];
    }
    const float inv0 = 1.f / L0, inv1 = 1.f / L1;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        f0[w] *= inv0;
        f1[w] *= inv1;
    }
    const bool has0 = 2 * c < G, has1 = 2 * c + 1 < G;  // padding heads are not written
    const size_t head0 = (size_t)b * H + kvh * G + 2 * c;
    const bool direct = n_part == 1;
    const size_t pi0 = head0 * prm.max_partitions + p, pi1 = pi0 + prm.max_partitions;
#pragma unroll
    for (int mt = 0; mt < S::kSteps; ++mt) {
        const int d = 16 * mt + g;
        float v00 = f0[0] * o[mt][0], v10 = f1[0] * o[mt][1];  // (head 2c, d), (head 2c+1, d)
        float v08 = f0[0] * o[mt][2], v18 = f1[0] * o[mt][3];  // ... at d + 8
#pragma unroll
        for (int w = 1; w < NW; ++w) {
            const float* rw = red + (w - 1) * kMaxGroup * S::kRedStride;
            v00 += f0[w] * rw[(2 * c) * S::kRedStride + d];
            v10 += f1[w] * rw[(2 * c + 1) * S::kRedStride + d];
            v08 += f0[w] * rw[(2 * c) * S::kRedStride + d + 8];
            v18 += f1[w] * rw[(2 * c + 1) * S::kRedStride + d + 8];
        }
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
            prm.max_logits[pi0] = M0;
            prm.exp_sums[pi0] = L0;
        }
        if (has1) {
            prm.max_logits[pi1] = M1;
            prm.exp_sums[pi1] = L1;
        }
    }
    }
    if (fused) fused_combine<D, NW>(prm, b, kvh, n_part, sm_abort + 1);  // a spare word of the control area
    PA_TRACE_MARK(4);
}

// ---------------------------------------------------------------------------
// Persistent schedule (PA_MODE_PERSISTENT).  pa_work_scan_kernel writes, per
// sequence, the exclusive prefix sum of its work items (work_items: one per
// (partition, kv head), one per kv head for an empty sequence, one for an
// invalid length) and resets the item counter.  A fixed grid of NW-warp CTAs
// (every CTA the SMs hold at once) takes items from that counter: CTA x
// starts with item x and then draws the next index with atomicAdd, so the
// last items end within about one item of each other whatever the length
// mix.  Sequence b of L tokens is cut into partitions of
// balanced_partition(L, P) tokens, the fewest of at most P evened out to
// whole blocks.
//
// Inside a CTA, warp w takes blocks w, w + NW, ... of every item, and its
// blocks form ONE stream across the CTA's items: stream position g uses the
// warp's stage g % NS and completes phase g / NS of that stage's mbarrier
// (initialised once per CTA, never again).  The copies run NS positions
// ahead of the math, into the next item when the current one ends, as far
// as the item indices are known: thread 0 draws item k + 2 while item k is
// processed and publishes it at the item's barrier.
//
// Each item ends with one CTA barrier: warps leave their (m, l, O) in a
// double-buffered merge area, and warp k % NW merges the item (in warp
// order 0..NW-1, so the bits do not depend on which warp merges) while the
// others go on to item k + 1.
// ---------------------------------------------------------------------------

// Work item i of the persistent schedule.  nblk = the blocks it streams:
// 0 for an invalid length, an empty sequence, or (never, with a work list
// built from the same lengths) a partition past the end.
struct PersistentItem {
    int b, p, kvh, L, part, nblk;
    bool bad;
};

// `offs` and `lens` are the work list and the lengths, in shared memory when
// the CTA cached them (persistent_seq_cache_bytes), else in global memory.
__device__ __forceinline__ PersistentItem persistent_item(const PartitionParams& prm, const int* offs,
                                                          const int* lens, int i) {
    int lo = 0, hi = prm.num_seqs;  // offs[lo] <= i < offs[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offs[mid] <= i)
            lo = mid;
        else
            hi = mid;
    }
    PersistentItem it;
    const int r = i - offs[lo];
    it.b = lo;
    it.p = r / prm.num_kv_heads;
    it.kvh = r % prm.num_kv_heads;
    it.L = lens[lo];
    it.bad = it.L < 0 || it.L > prm.max_seq_len || it.L > prm.max_blocks_per_seq * kBlockSize;
    it.part = balanced_partition(it.L, prm.partition_size);
    it.nblk = 0;
    if (!it.bad && it.L > 0) {
        const int bpp = it.part / kBlockSize;
        it.nblk = max(0, min(bpp, (it.L + kBlockSize - 1) / kBlockSize - it.p * bpp));
    }
    return it;
}

// Shared memory of a persistent CTA: the NW x NS stages, then two merge areas
// ([NW][8 heads][D + 4] floats each, with per-warp max and exp sum), the
// mbarriers, the published item indices and the abort flag; a batch of at
// most kPersistentSeqCache sequences adds its work list and lengths
// (persistent_seq_cache_bytes) after kSmemBytes - 1024.
template <int D, int NW, int NS>
struct PersistentShape {
    using P = PartitionShape<D, NW, NS>;
    // a one-warp CTA merges nothing: no merge areas
    static constexpr int kRedFloats = NW > 1 ? NW * kMaxGroup * P::kRedStride : 0;
    static constexpr int kStatFloats = NW > 1 ? 2 * NW * kMaxGroup : 0;
    static constexpr int kRedArea = P::kStageArea;                  // offset of the merge areas
    static constexpr int kStatArea = kRedArea + 2 * kRedFloats * 4;  // [2][NW][8] max, then exp sums
    static constexpr int kBarArea = kStatArea + 2 * kStatFloats * 4;  // NW * NS mbarriers
    static constexpr int kCtrlArea = kBarArea + NW * NS * 8;                 // 4 item indices, abort flag
    static constexpr int kSmemBytes = 1024 + kCtrlArea + 32;
    static_assert(kBarArea % 8 == 0, "mbarrier alignment");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget of one CTA");
};

template <int D, int NW, int NS>
__global__ void __launch_bounds__(NW * 32, 1)
    pa_partition_persistent_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                   const __grid_constant__ CUtensorMap tmap_v, const PartitionParams prm) {
    using S = PartitionShape<D, NW, NS>;
    using Q = PersistentShape<D, NW, NS>;
    // the work list and the item counter are written by the preceding (scan) grid
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    float* red = reinterpret_cast<float*>(smem + Q::kRedArea);    // [2][NW][8][kRedStride]
    float* st_m = reinterpret_cast<float*>(smem + Q::kStatArea);  // [2][NW][8]
    float* st_l = st_m + 2 * NW * kMaxGroup;                      // [2][NW][8]
    int* items = reinterpret_cast<int*>(smem + Q::kCtrlArea);     // CTA-local item k -> index, k mod 4
    int* sm_abort = items + 4;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = prm.group, H = prm.num_heads;
    const uint32_t stage0 = smem_addr(smem) + warp * NS * S::kStageBytes;
    const uint32_t bar0 = smem_addr(smem) + Q::kBarArea + warp * NS * 8;
    // Items are located by binary search over the work list, on the copy
    // side and again at the start of each item's math: from shared memory
    // when the batch is small enough to cache.
    const int* offs = prm.work_offsets;
    const int* lens = prm.seq_lens;
    if (prm.num_seqs <= kPersistentSeqCache) {
        int* so = reinterpret_cast<int*>(smem + Q::kSmemBytes - 1024);
        int* sl = so + prm.num_seqs + 1;
        for (int x = threadIdx.x; x <= prm.num_seqs; x += blockDim.x) so[x] = __ldg(prm.work_offsets + x);
        for (int x = threadIdx.x; x < prm.num_seqs; x += blockDim.x) sl[x] = __ldg(prm.seq_lens + x);
        offs = so;
        lens = sl;
    }
    const int total = __ldg(prm.work_offsets + prm.num_seqs);

    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8 * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        items[0] = blockIdx.x;
        items[1] = (int)blockIdx.x < total ? atomicAdd(prm.work_counter, 1) : total;
        *sm_abort = 0;
    }
    __syncthreads();

    // ---- copy side: this warp's blocks of the CTA's items, in order ----
    int is_k = 0;         // CTA-local item being copied
    bool is_dec = false;  // its blocks are known
    int is_j = 0, is_nblk = 0, is_kvh = 0, is_ids = -1;
    const int32_t* is_bt = prm.block_tables;
    uint32_t issued = 0;      // stream positions issued so far
    uint32_t valid_bits = 0;  // stage s holds a block with a legal id
    // Issue the next stream position if its item index is published
    // (CTA-local items up to `known`); warp-uniform.
    auto issue_next = [&](int known) {
        for (;;) {
            if (is_dec) {
                if (is_j < is_nblk) break;
                ++is_k;
                is_dec = false;
            }
            if (is_k > known) return;
            const int I = items[is_k & 3];
            if (I >= total) return;
            const PersistentItem it = persistent_item(prm, offs, lens, I);
            is_nblk = it.nblk;
            is_kvh = it.kvh;
            is_j = warp;
            is_bt = prm.block_tables + (size_t)it.b * prm.max_blocks_per_seq + it.p * (it.part / kBlockSize);
            is_dec = true;
        }
        // the warp's t-th block of the item; block ids 32 at a time, only
        // below the sequence's last block
        const int t = (is_j - warp) / NW;
        if ((t & 31) == 0) {
            const int jj = warp + NW * (t + lane);
            is_ids = jj < is_nblk ? __ldg(is_bt + jj) : -1;
        }
        const int phys = __shfl_sync(kFull, is_ids, t & 31);
        const int s = (int)(issued % NS);
        const uint32_t bar = bar0 + 8 * s;
        const bool ok = phys >= 0 && (long long)phys < prm.num_blocks;
        valid_bits = ok ? (valid_bits | (1u << s)) : (valid_bits & ~(1u << s));
        if (lane == 0) {
            if (ok) {
                mbar_arrive_expect_tx(bar, S::kStageBytes);
                const int row = (phys * prm.num_kv_heads + is_kvh) * kBlockSize;
                const uint32_t kdst = stage0 + s * S::kStageBytes;
                tma_load_3d(kdst, &tmap_k, 0, row, 0, bar);
                tma_load_3d(kdst + S::kTileBytes, &tmap_v, 0, row, 0, bar);
            } else {
                atomicOr(&g_status, PA_DEV_BAD_BLOCK_ID);
                mbar_arrive(bar);  // complete the phase so the math stays in step
            }
        }
        is_j += NW;
        ++issued;
    };
    for (int x = 0; x < NS; ++x) issue_next(1);

    // ---- math side ----
    const int g = lane >> 2, c = lane & 3;  // MMA fragment row group / column pair
    const float sl2 = prm.scale_log2;
    uint32_t pos = 0;  // stream position of the warp's next block
    for (int k = 0;; ++k) {
        const int I = items[k & 3];
        if (I >= total) break;  // the same for every warp
        const PersistentItem it = persistent_item(prm, offs, lens, I);
        // thread 0 draws the index of item k + 2 now; it is published at this item's barrier
        int drawn = total;
        if (threadIdx.x == 0 && items[(k + 1) & 3] < total) drawn = atomicAdd(prm.work_counter, 1);
        const int blk0 = it.p * (it.part / kBlockSize);

        float o[S::kSteps][4];
#pragma unroll
        for (int x = 0; x < S::kSteps; ++x) o[x][0] = o[x][1] = o[x][2] = o[x][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        if (warp < it.nblk) {
            uint32_t qb[S::kSteps][2];
            const int hq = g < G ? g : 0;  // lanes of padding heads load nothing
            const uint32_t* qrow =
                reinterpret_cast<const uint32_t*>(prm.q + ((size_t)it.b * H + it.kvh * G + hq) * D);
#pragma unroll
            for (int ks = 0; ks < S::kSteps; ++ks) {
                qb[ks][0] = g < G ? __ldg(qrow + 8 * ks + c) : 0u;
                qb[ks][1] = g < G ? __ldg(qrow + 8 * ks + 4 + c) : 0u;
            }
            for (int j = warp; j < it.nblk; j += NW, ++pos) {
                const int s = (int)(pos % NS);
                if (prm.force_timeout || !mbar_wait(bar0 + 8 * s, (pos / NS) & 1, prm.wait_limit)) {
                    // drain this warp's copies, report, and end the CTA at the barrier below
                    for (uint32_t x = pos; x < issued; ++x)
                        mbar_wait(bar0 + 8 * (x % NS), (x / NS) & 1, kDefaultWaitLimit);
                    pos = issued;
                    if (lane == 0) {
                        atomicOr(&g_status, PA_DEV_TIMEOUT);
                        atomicExch(sm_abort, 1);
                    }
                    break;
                }
                if ((valid_bits >> s) & 1u) {
                    const uint32_t kst = stage0 + s * S::kStageBytes;
                    warp_block_update<D>(qb, o, m0, m1, l0, l1, kst, kst + S::kTileBytes,
                                         smem + (kst + S::kTileBytes - smem_addr(smem)),
                                         min(kBlockSize, it.L - (blk0 + j) * kBlockSize), sl2);
                }
                __syncwarp();
                issue_next(k + 1);  // the stage just read takes position pos + NS
            }
        }
        // exp sums: add the shares of the 8 lanes holding the same heads
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(kFull, l0, off);
            l1 += __shfl_xor_sync(kFull, l1, off);
        }
        const int merger = k % NW, buf = k & 1;
        if (warp != merger && warp < it.nblk) {
            float* rw = red + (buf * NW + warp) * kMaxGroup * S::kRedStride;
#pragma unroll
            for (int mt = 0; mt < S::kSteps; ++mt) {
                const int d = 16 * mt + g;
                rw[(2 * c) * S::kRedStride + d] = o[mt][0];
                rw[(2 * c + 1) * S::kRedStride + d] = o[mt][1];
                rw[(2 * c) * S::kRedStride + d + 8] = o[mt][2];
                rw[(2 * c + 1) * S::kRedStride + d + 8] = o[mt][3];
            }
            if (g == 0) {
                st_m[(buf * NW + warp) * kMaxGroup + 2 * c] = m0;
                st_m[(buf * NW + warp) * kMaxGroup + 2 * c + 1] = m1;
                st_l[(buf * NW + warp) * kMaxGroup + 2 * c] = l0;
                st_l[(buf * NW + warp) * kMaxGroup + 2 * c + 1] = l1;
            }
        }
        if (threadIdx.x == 0) items[(k + 2) & 3] = drawn;
        __syncthreads();
        if (*sm_abort) break;  // the same for every warp
        // top the copies up to NS ahead: item k + 2 is known now
        for (int x = 0; x < NS && issued - pos < (uint32_t)NS; ++x) issue_next(k + 2);
        if (warp != merger) continue;

        // ---- merger warp: item k's output ----
        if (it.bad) {
            if (lane == 0) atomicOr(&g_status, PA_DEV_BAD_SEQ_LEN);
            continue;
        }
        if (it.L == 0) {  // empty sequence: its G heads of this kv head are zero
            for (int x = lane; x < G * D; x += 32)
                prm.out[((size_t)it.b * H + it.kvh * G) * D + x] = __float2half_rn(0.f);
            continue;
        }
        if (it.nblk == 0) continue;
        // warps w < nw streamed blocks; the merger's own state is in registers,
        // the others' in merge area `buf`.  M = max m_w, f_w = 2^(m_w - M) / L
        // with L = sum_w 2^(m_w - M) l_w, summed in warp order.
        const int nw = min(NW, it.nblk);
        const float* sm = st_m + buf * NW * kMaxGroup;
        const float* sl = st_l + buf * NW * kMaxGroup;
        float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            if (w >= nw) continue;
            M0 = fmaxf(M0, w == merger ? m0 : sm[w * kMaxGroup + 2 * c]);
            M1 = fmaxf(M1, w == merger ? m1 : sm[w * kMaxGroup + 2 * c + 1]);
        }
        float f0[NW], f1[NW];
        float L0 = 0.f, L1 = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            f0[w] = f1[w] = 0.f;
            if (w >= nw) continue;
            const float mw0 = w == merger ? m0 : sm[w * kMaxGroup + 2 * c];
            const float mw1 = w == merger ? m1 : sm[w * kMaxGroup + 2 * c + 1];
            f0[w] = mw0 == -INFINITY ? 0.f : exp2f(mw0 - M0);
            f1[w] = mw1 == -INFINITY ? 0.f : exp2f(mw1 - M1);
            L0 += f0[w] * (w == merger ? l0 : sl[w * kMaxGroup + 2 * c]);
            L1 += f1[w] * (w == merger ? l1 : sl[w * kMaxGroup + 2 * c + 1]);
        }
        const float inv0 = 1.f / L0, inv1 = 1.f / L1;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            f0[w] *= inv0;
            f1[w] *= inv1;
        }
        const int n_part = (it.L + it.part - 1) / it.part;
        const bool has0 = 2 * c < G, has1 = 2 * c + 1 < G;  // padding heads are not written
        const size_t head0 = (size_t)it.b * H + it.kvh * G + 2 * c;
        const bool direct = n_part == 1;
        const size_t pi0 = head0 * prm.max_partitions + it.p, pi1 = pi0 + prm.max_partitions;
#pragma unroll
        for (int mt = 0; mt < S::kSteps; ++mt) {
            const int d = 16 * mt + g;
            float v00 = 0.f, v10 = 0.f, v08 = 0.f, v18 = 0.f;  // (head 2c, d), (2c+1, d), then d + 8
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                if (w >= nw) continue;
                if (w == merger) {
                    v00 += f0[w] * o[mt][0];
                    v10 += f1[w] * o[mt][1];
                    v08 += f0[w] * o[mt][2];
                    v18 += f1[w] * o[mt][3];
                } else {
                    const float* rw = red + (buf * NW + w) * kMaxGroup * S::kRedStride;
                    v00 += f0[w] * rw[(2 * c) * S::kRedStride + d];
                    v10 += f1[w] * rw[(2 * c + 1) * S::kRedStride + d];
                    v08 += f0[w] * rw[(2 * c) * S::kRedStride + d + 8];
                    v18 += f1[w] * rw[(2 * c + 1) * S::kRedStride + d + 8];
                }
            }
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
                prm.max_logits[pi0] = M0;
                prm.exp_sums[pi0] = L0;
            }
            if (has1) {
                prm.max_logits[pi1] = M1;
                prm.exp_sums[pi1] = L1;
            }
        }
    }
    // copies issued ahead of an abort complete before the CTA exits
    for (uint32_t x = pos; x < issued; ++x) mbar_wait(bar0 + 8 * (x % NS), (x / NS) & 1, kDefaultWaitLimit);
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
template <int D, int W>
__global__ void __launch_bounds__(kReduceThreads) pa_reduce_kernel(const ReduceParams prm) {
    constexpr int kLanes = W / 4;                    // float4 columns of a slice
    constexpr int kGroups = kReduceThreads / kLanes; // partition groups
    static_assert(W <= D && D % W == 0 && kLanes <= kReduceThreads, "slice width");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int h = blockIdx.x, b = blockIdx.y, slice = blockIdx.z;
    const int L = prm.seq_lens[b];
    // single-partition, empty and invalid sequences were finished by the partition kernel
    if (L <= prm.partition_size || L > prm.max_seq_len || L > prm.max_blocks_per_seq * kBlockSize) return;
    const int part = prm.balanced ? balanced_partition(L, prm.partition_size) : prm.partition_size;
    const int n = (L + part - 1) / part;
    const size_t base = ((size_t)b * prm.num_heads + h) * prm.max_partitions;
    const float* ml = prm.max_logits + base;
    const float* el = prm.exp_sums + base;

    __shared__ float4 red_acc[kGroups][kLanes];
    __shared__ float red_m[kGroups];
    __shared__ float red_w[kGroups];

    const int col = threadIdx.x % kLanes, pg = threadIdx.x / kLanes;
    const float4* tp = reinterpret_cast<const float4*>(prm.tmp_out + base * D + slice * W) + col;
    float m = -INFINITY, wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int p = pg; p < n; p += kGroups) {
        const float mp = ml[p], lp = el[p];
        const float4 t = tp[(size_t)p * (D / 4)];
        const float mn = fmaxf(m, mp);
        const float alpha = exp2f(m - mn);  // 0 on the first partition (m = -inf)
        const float beta = lp * exp2f(mp - mn);
        wsum = wsum * alpha + beta;
        acc.x = acc.x * alpha + beta * t.x;
        acc.y = acc.y * alpha + beta * t.y;
        acc.z = acc.z * alpha + beta * t.z;
        acc.w = acc.w * alpha + beta * t.w;
        m = mn;
    }
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

template <int D, int NW, int NS>
cudaError_t launch_partition_t(const PartitionParams& prm, const CUtensorMap& tk, const CUtensorMap& tv, dim3 grid,
                               cudaStream_t stream) {
    const int smem = PartitionShape<D, NW, NS>::kSmemBytes;
    // The attribute is per device; setting it on every call costs little and
    // keeps multi-device processes correct.
    cudaError_t e =
        cudaFuncSetAttribute(pa_partition_kernel<D, NW, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, pa_partition_kernel<D, NW, NS>, tk, tv, prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D, int W>
cudaError_t launch_reduce_t(const ReduceParams& prm, dim3 grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kReduceThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, pa_reduce_kernel<D, W>, prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_reduce_d(int width, const ReduceParams& prm, dim3 grid, cudaStream_t stream) {
    switch (width) {
        case 32: return launch_reduce_t<D, 32>(prm, grid, stream);
        case 64: return launch_reduce_t<D, 64>(prm, grid, stream);
        case 128: if constexpr (D >= 128) return launch_reduce_t<D, 128>(prm, grid, stream); else break;
        case 256: if constexpr (D >= 256) return launch_reduce_t<D, 256>(prm, grid, stream); else break;
        default: break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_partition(int head_dim, int warps, int stages, const PartitionParams& prm, const CUtensorMap& tk,
                             const CUtensorMap& tv, dim3 grid, cudaStream_t stream) {
#define PA_LAUNCH_CASE(W_, S_)                                                          \
    if (warps == W_ && stages == S_) {                                                 \
        switch (head_dim) {                                                            \
            case 64: return launch_partition_t<64, W_, S_>(prm, tk, tv, grid, stream);   \
            case 128: return launch_partition_t<128, W_, S_>(prm, tk, tv, grid, stream); \
            case 256: return launch_partition_t<256, W_, S_>(prm, tk, tv, grid, stream); \
            default: return cudaErrorInvalidValue;                                     \
        }                                                                              \
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

// The persistent kernel's CTA shapes (warps, stages per warp).
#define PA_FOR_EACH_PERSISTENT_SHAPE(X) X(1, 2) X(2, 2) X(4, 2)

int persistent_smem_bytes(int head_dim, int warps, int stages) {
#define PA_PSMEM_CASE(W_, S_)                                                         \
    if (warps == W_ && stages == S_) {                                               \
        switch (head_dim) {                                                          \
            case 64: return PersistentShape<64, W_, S_>::kSmemBytes;                 \
            case 128: return PersistentShape<128, W_, S_>::kSmemBytes;               \
            case 256: return PersistentShape<256, W_, S_>::kSmemBytes;               \
            default: return -1;                                                      \
        }                                                                            \
    }
    PA_FOR_EACH_PERSISTENT_SHAPE(PA_PSMEM_CASE)
#undef PA_PSMEM_CASE
    return -1;
}

namespace {
template <int D, int NW, int NS>
cudaError_t launch_persistent_t(const PartitionParams& prm, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                                cudaStream_t stream) {
    const int smem = PersistentShape<D, NW, NS>::kSmemBytes + persistent_seq_cache_bytes(prm.num_seqs);
    cudaError_t e = cudaFuncSetAttribute(pa_partition_persistent_kernel<D, NW, NS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, pa_partition_persistent_kernel<D, NW, NS>, tk, tv, prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_partition_persistent(int head_dim, int warps, int stages, const PartitionParams& prm,
                                        const CUtensorMap& tk, const CUtensorMap& tv, int grid, cudaStream_t stream) {
    if (!prm.work_offsets || !prm.work_counter || grid <= 0) return cudaErrorInvalidValue;
#define PA_PLAUNCH_CASE(W_, S_)                                                              \
    if (warps == W_ && stages == S_) {                                                      \
        switch (head_dim) {                                                                 \
            case 64: return launch_persistent_t<64, W_, S_>(prm, tk, tv, grid, stream);     \
            case 128: return launch_persistent_t<128, W_, S_>(prm, tk, tv, grid, stream);   \
            case 256: return launch_persistent_t<256, W_, S_>(prm, tk, tv, grid, stream);   \
            default: return cudaErrorInvalidValue;                                          \
        }                                                                                   \
    }
    PA_FOR_EACH_PERSISTENT_SHAPE(PA_PLAUNCH_CASE)
#undef PA_PLAUNCH_CASE
    return cudaErrorInvalidValue;
}

// Exclusive prefix sums of the per-sequence work items (one CTA of 1024
// threads; each thread sums a contiguous run of sequences, then the runs are
// scanned across the block).
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads) pa_work_scan_kernel(const ScanParams prm) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ int warp_sums[kScanThreads / 32];
    const int per = (prm.num_seqs + kScanThreads - 1) / kScanThreads;
    const int b0 = threadIdx.x * per, b1 = min(prm.num_seqs, b0 + per);
    int local = 0;
    for (int b = b0; b < b1; ++b)
        local += work_items(__ldg(prm.seq_lens + b), prm.max_seq_len, prm.max_blocks_per_seq, prm.partition_size,
                            prm.num_kv_heads);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(kFull, w, off);
            if (lane >= off) w += v;
        }
        warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    int run = incl - local + (warp > 0 ? warp_sums[warp - 1] : 0);  // exclusive start of this thread's run
    for (int b = b0; b < b1; ++b) {
        prm.work_offsets[b] = run;
        run += work_items(__ldg(prm.seq_lens + b), prm.max_seq_len, prm.max_blocks_per_seq, prm.partition_size,
                          prm.num_kv_heads);
    }
    if (threadIdx.x == kScanThreads - 1) {
        prm.work_offsets[prm.num_seqs] = warp_sums[kScanThreads / 32 - 1];
        *prm.work_counter = prm.first_dynamic;  // items below it are taken by CTA index
    }
}

cudaError_t launch_work_scan(const ScanParams& prm, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kScanThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, pa_work_scan_kernel, prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
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
