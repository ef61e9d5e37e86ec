// Pieces shared by the decode partition kernels (pa_kernels.cu: one CTA per
// (partition, kv head, sequence); pa_persistent.cu: the persistent schedule):
// the shared-memory shape of a CTA and the per-block online-softmax update
// of one warp.  See pa_kernels.cu for the hardware mapping.
#pragma once

#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

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

}  // namespace pa
