// Persistent schedule of the decode partition work (PA_MODE_PERSISTENT):
// pa_work_scan_kernel builds the work list on the device, and
// pa_partition_persistent_kernel walks it with a fixed grid.  The per-block
// math is the grid kernel's (pa_partition_block.cuh).
#include "pa_internal.h"

#include <math.h>

#include "pa_decode.h"
#include "pa_device.cuh"
#include "pa_partition_block.cuh"

namespace pa {

// ---------------------------------------------------------------------------
// Persistent schedule (PA_MODE_PERSISTENT).  pa_work_scan_kernel sizes each
// sequence's partitions, orders the sequences longest partition first and
// writes the exclusive prefix sums of their work items in that order (one
// item per (partition, kv head), one per kv head for an empty sequence, one
// for an invalid length), then resets the item counter.  Without a caller's
// partition size, the partitions are apportioned: with slots = grid / kv
// heads, the scan finds the smallest cap S (blocks per partition) for which
// the batch's partitions -- ceil(blocks_b / S) per sequence -- fit the
// slots, so the items fill one wave and the longest is as short as one wave
// allows; with at least as many sequences as slots, S = total blocks / slots.
// A fixed grid of NW-warp CTAs (every CTA the SMs hold at once) takes items
// from that counter: CTA x starts with item x and then draws the next index
// with atomicAdd, so the last items -- the shortest, by the order -- end
// within about one item of each other.
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

// Work item i of the persistent schedule: blocks blk0 .. blk0 + nblk - 1 of
// sequence b for kv head kvh.  nblk = 0 for an invalid length, an empty
// sequence, or (never, with a work list built from the same lengths) a
// partition past the end.  The item's partial goes to slot `slot` of its
// (sequence, head) rows, or straight to the output when the sequence has no
// other item (`direct`).
struct PersistentItem {
    int b, kvh, L, blk0, nblk, slot;
    bool bad, direct;
};

// The schedule's tables (work list over the schedule order, the order, the
// lengths and the partition sizes), in shared memory when the CTA cached them
// (persistent_seq_cache_bytes), else in global memory.
struct ScheduleTables {
    const int* offs;
    const int* order;
    const int* lens;
    const int* parts;
};

__device__ __forceinline__ PersistentItem persistent_item(const PartitionParams& prm, const ScheduleTables& tb, int i) {
    int lo = 0, hi = prm.num_seqs;  // offs[lo] <= i < offs[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tb.offs[mid] <= i)
            lo = mid;
        else
            hi = mid;
    }
    PersistentItem it;
    const int r = i - tb.offs[lo];
    it.b = tb.order[lo];
    const int p = r / prm.num_kv_heads;
    it.kvh = r % prm.num_kv_heads;
    it.L = tb.lens[it.b];
    it.bad = it.L < 0 || it.L > prm.max_seq_len || it.L > prm.max_blocks_per_seq * kBlockSize;
    const int part = tb.parts[it.b];
    const int bpp = part / kBlockSize;
    it.blk0 = p * bpp;
    it.slot = p;
    it.nblk = 0;
    it.direct = false;
    if (!it.bad && it.L > 0) {
        it.nblk = max(0, min(bpp, (it.L + kBlockSize - 1) / kBlockSize - it.blk0));
        it.direct = it.L <= part;  // one partition
    }
    return it;
}

// ---------------------------------------------------------------------------
// Flat one-wave split (PA_MODE_FLAT): no work list.  Every CTA reads the
// batch's lengths, and with nb_b = ceil(L_b / 16) blocks per valid sequence,
// S_b their exclusive prefix sums and T = S_B, CTA c of the C CTAs of a kv
// head (C' = min(C, T) of them busy) streams blocks [f(c), f(c + 1)) of the
// batch's concatenated block list, f(c) = floor(c T / C').  Each sequence
// that range meets is one item: its blocks j0 .. j1 - 1, with slot
// c - c_first(b) of the sequence's partials, c_first(b) = the CTA whose range
// holds the sequence's first block; a sequence met by one CTA only is written
// straight to the output.  Every CTA streams T / C' blocks (+-1), whatever
// the lengths, so the wave has no ragged tail of short and long CTAs.
// ---------------------------------------------------------------------------

// The flat split's CTA range start f(c) and the CTA holding block `pos`.
__device__ __forceinline__ int flat_start(int c, int T, int C) { return (int)(((long long)c * T) / C); }
__device__ __forceinline__ int flat_cta_of(int pos, int T, int C) {
    int c = (int)(((long long)pos * C) / T);
    while (c + 1 < C && flat_start(c + 1, T, C) <= pos) ++c;
    return c;
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

// Diagnostic builds (-DPA_TRACE): per-CTA records in the decode timeline's
// format {sm id, entry, first block ready, first item done, exit}
// (global-timer ns).
#ifdef PA_TRACE
#define PA_PT_MARK(slot)                                                      \
    do {                                                                      \
        if (prm.trace && threadIdx.x == 0) {                                  \
            unsigned long long g_;                                            \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g_));           \
            prm.trace[(size_t)blockIdx.x * 5 + (slot)] = g_;                  \
        }                                                                     \
    } while (0)
#else
#define PA_PT_MARK(slot) \
    do {                 \
    } while (0)
#endif

template <int D, int NW, int NS, bool Flat>
__global__ void __launch_bounds__(NW * 32, 1)
    pa_partition_persistent_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                   const __grid_constant__ CUtensorMap tmap_v, const PartitionParams prm) {
    using S = PartitionShape<D, NW, NS>;
    using Q = PersistentShape<D, NW, NS>;
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
    // the copy barriers and the tensor maps' descriptors read nothing the
    // preceding grids write: set up before the dependency wait
    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8 * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_v)) : "memory");
    }

    // the work list and the item counter are written by the preceding (scan) grid
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
#ifdef PA_TRACE
    if (prm.trace && threadIdx.x == 0) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        prm.trace[(size_t)blockIdx.x * 5] = smid;
    }
#endif
    PA_PT_MARK(1);

    // Items are located by binary search over the work list, on the copy
    // side and again at the start of each item's math: from shared memory
    // when the batch is small enough to cache.
    ScheduleTables tb{prm.work_offsets, prm.seq_order, prm.seq_lens, prm.part_sizes};
    // Flat split: this CTA's kv head, its place c among the C CTAs of that kv
    // head, the busy CTAs Cb = min(C, T), its block range [f_lo, f_hi), and in
    // shared memory the lengths, the block prefix sums and its items (the
    // sequences its range meets)
    int f_kvh = 0, f_c = 0, f_T = 0, f_Cb = 0, f_lo = 0, f_hi = 0;
    const int* f_len = nullptr;
    const int* f_S = nullptr;
    const int* f_items = nullptr;
    int total = 0;
    if constexpr (Flat) {
        const int B = prm.num_seqs;  // at most kPersistentSeqCache (the host checks)
        int* sl = reinterpret_cast<int*>(smem + Q::kSmemBytes - 1024);
        int* sS = sl + B;      // [B + 1]
        int* sI = sS + B + 1;  // [B + 1]: the items, then their count
        for (int x = threadIdx.x; x < B; x += blockDim.x) {
            const int L = __ldg(prm.seq_lens + x);
            sl[x] = L;
            const bool ok = L > 0 && L <= prm.max_seq_len && L <= prm.max_blocks_per_seq * kBlockSize;
            sS[x + 1] = ok ? (L + kBlockSize - 1) / kBlockSize : 0;
        }
        __syncthreads();
        if (warp == 0) {  // inclusive scan of the block counts, 32 at a time
            int run = 0;
            if (lane == 0) sS[0] = 0;
            for (int base = 0; base < B; base += 32) {
                const int x = base + lane;
                int v = x < B ? sS[x + 1] : 0;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int u = __shfl_up_sync(kFull, v, off);
                    if (lane >= off) v += u;
                }
                if (x < B) sS[x + 1] = run + v;
                run += __shfl_sync(kFull, v, 31);
            }
        }
        __syncthreads();
        const int C = prm.max_partitions;  // CTAs per kv head
        f_kvh = (int)blockIdx.x % prm.num_kv_heads;
        f_c = (int)blockIdx.x / prm.num_kv_heads;
        f_T = sS[B];
        f_Cb = min(C, f_T);
        if (f_c < f_Cb) {
            f_lo = flat_start(f_c, f_T, f_Cb);
            f_hi = flat_start(f_c + 1, f_T, f_Cb);
        }
        if (threadIdx.x == 0) {
            int n = 0;
            if (f_c < f_Cb) {
                int a = 0, z = B;  // the first sequence whose blocks end past f_lo
                while (a < z) {
                    const int mid = (a + z) >> 1;
                    if (sS[mid + 1] > f_lo)
                        z = mid;
                    else
                        a = mid + 1;
                }
                for (int b = a; b < B && sS[b] < f_hi; ++b) {
                    if (sS[b + 1] == sS[b]) continue;  // no blocks
                    sI[n++] = b;
                    // the CTA with a sequence's first block records its partial count
                    if (prm.part_counts && f_kvh == 0 && sS[b] >= f_lo)
                        prm.part_counts[b] = flat_cta_of(sS[b + 1] - 1, f_T, f_Cb) - f_c + 1;
                }
            }
            sI[B] = n;
        }
        // empty sequences: zero output (CTA b % C of each kv head); invalid
        // lengths: reported once
        for (int b = f_c; b < B; b += C) {
            if (sl[b] == 0)
                for (int x = threadIdx.x; x < G * D; x += blockDim.x)
                    prm.out[((size_t)b * H + f_kvh * G) * D + x] = __float2half_rn(0.f);
        }
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            for (int b = 0; b < B; ++b)
                if (sl[b] < 0 || sl[b] > prm.max_seq_len || sl[b] > prm.max_blocks_per_seq * kBlockSize) {
                    atomicOr(prm.status, PA_DEV_BAD_SEQ_LEN);
                    break;
                }
        }
        __syncthreads();
        total = sI[B];
        f_len = sl;
        f_S = sS;
        f_items = sI;
    } else if (prm.num_seqs <= kPersistentSeqCache) {
        const int B = prm.num_seqs;
        int* so = reinterpret_cast<int*>(smem + Q::kSmemBytes - 1024);
        int *sr = so + B + 1, *sl = sr + B, *sp = sl + B;
        for (int x = threadIdx.x; x <= B; x += blockDim.x) so[x] = __ldg(prm.work_offsets + x);
        for (int x = threadIdx.x; x < B; x += blockDim.x) {
            sr[x] = __ldg(prm.seq_order + x);
            sl[x] = __ldg(prm.seq_lens + x);
            sp[x] = __ldg(prm.part_sizes + x);
        }
        tb = ScheduleTables{so, sr, sl, sp};
    }
    if constexpr (!Flat) total = __ldg(prm.work_offsets + prm.num_seqs);

    // Item I of this CTA's schedule (a work-list index, or for the flat split
    // an index into this CTA's own items)
    auto item_at = [&](int I) -> PersistentItem {
        if constexpr (Flat) {
            PersistentItem it;
            it.b = f_items[I];
            it.kvh = f_kvh;
            it.L = f_len[it.b];
            it.bad = false;
            const int S0 = f_S[it.b], S1 = f_S[it.b + 1];
            it.blk0 = max(f_lo, S0) - S0;
            it.nblk = min(f_hi, S1) - S0 - it.blk0;
            const int first = S0 >= f_lo ? f_c : flat_cta_of(S0, f_T, f_Cb);
            it.slot = f_c - first;
            it.direct = first == f_c && S1 <= f_hi;  // no other CTA meets this sequence
            return it;
        } else {
            return persistent_item(prm, tb, I);
        }
    };

    if (threadIdx.x == 0) {
        if constexpr (Flat) {
            items[0] = 0;
            items[1] = 1;
        } else {
            items[0] = blockIdx.x;
            items[1] = (int)blockIdx.x < total ? atomicAdd(prm.work_counter, 1) : total;
        }
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
            const PersistentItem it = item_at(I);
            is_nblk = it.nblk;
            is_kvh = it.kvh;
            is_j = warp;
            is_bt = prm.block_tables + (size_t)it.b * prm.max_blocks_per_seq + it.blk0;
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
                atomicOr(prm.status, PA_DEV_BAD_BLOCK_ID);
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
        const PersistentItem it = item_at(I);
        // thread 0 draws the index of item k + 2 now; it is published at this item's barrier
        int drawn = total;
        if constexpr (Flat) {
            drawn = k + 2;
        } else {
            if (threadIdx.x == 0 && items[(k + 1) & 3] < total) drawn = atomicAdd(prm.work_counter, 1);
        }
        const int blk0 = it.blk0;

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
                        atomicOr(prm.status, PA_DEV_TIMEOUT);
                        atomicExch(sm_abort, 1);
                    }
                    break;
                }
                if (k == 0 && j == warp) PA_PT_MARK(2);
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
        const int buf = k & 1;
        if (NW > 1 && warp < it.nblk) {  // warps with blocks leave (m, l, O) in merge area buf
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
        if (k == 0) PA_PT_MARK(3);
        if (threadIdx.x == 0) items[(k + 2) & 3] = drawn;
        __syncthreads();
        if (*sm_abort) break;  // the same for every warp
        // top the copies up to NS ahead: item k + 2 is known now
        for (int x = 0; x < NS && issued - pos < (uint32_t)NS; ++x) issue_next(k + 2);

        // ---- item k's output ----
        if (it.bad) {
            if (warp == 0 && lane == 0) atomicOr(prm.status, PA_DEV_BAD_SEQ_LEN);
            continue;
        }
        if (it.L == 0) {  // empty sequence: its G heads of this kv head are zero
            for (int x = threadIdx.x; x < G * D; x += NW * 32)
                prm.out[((size_t)it.b * H + it.kvh * G) * D + x] = __float2half_rn(0.f);
            continue;
        }
        if (it.nblk == 0) continue;
        const bool direct = it.direct;
        if constexpr (NW == 1) {
            // one warp: o / l straight from the MMA fragments (lane (g, c)
            // holds heads 2c, 2c + 1); a partition whose blocks all had
            // illegal ids (m = -inf) was reported when they were copied
            const float w0 = m0 == -INFINITY ? 0.f : 1.f, w1 = m1 == -INFINITY ? 0.f : 1.f;
            const float L0 = w0 * l0, L1 = w1 * l1;
            const float f0 = w0 * (1.f / L0), f1 = w1 * (1.f / L1);
            const bool has0 = 2 * c < G, has1 = 2 * c + 1 < G;  // padding heads are not written
            const size_t head0 = (size_t)it.b * H + it.kvh * G + 2 * c;
            const size_t pi0 = head0 * prm.max_partitions + it.slot, pi1 = pi0 + prm.max_partitions;
#pragma unroll
            for (int mt = 0; mt < S::kSteps; ++mt) {
                const int d = 16 * mt + g;
                const float v00 = f0 * o[mt][0], v10 = f1 * o[mt][1], v08 = f0 * o[mt][2], v18 = f1 * o[mt][3];
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
            // every warp merges dims [w D/NW, (w+1) D/NW) of every head from
            // merge area buf (lane (h, q): head h, dim pairs 2q, 2q + 1 of each
            // 8-dim group), summing in warp order over the nw warps that had
            // blocks: M = max m_w, f_w = 2^(m_w - M) / L, L = sum_w 2^(m_w - M) l_w
            constexpr int kSlice = D / NW;
            static_assert(kSlice % 8 == 0, "a warp merges whole 8-dim groups");
            const int nw = min(NW, it.nblk);
            const float* sm = st_m + buf * NW * kMaxGroup;
            const float* sl = st_l + buf * NW * kMaxGroup;
            const float* rb = red + buf * NW * kMaxGroup * S::kRedStride;
            const int h = lane >> 2, qd = lane & 3;
            if (h < G) {  // padding heads are not written
                float Mh = sm[h];
#pragma unroll
                for (int w = 1; w < NW; ++w)
                    if (w < nw) Mh = fmaxf(Mh, sm[w * kMaxGroup + h]);
                float f[NW];
                f[0] = sm[h] == -INFINITY ? 0.f : exp2f(sm[h] - Mh);
                float Lh = f[0] * sl[h];
#pragma unroll
                for (int w = 1; w < NW; ++w) {
                    f[w] = 0.f;
                    if (w < nw) {
                        const float mw = sm[w * kMaxGroup + h];
                        f[w] = mw == -INFINITY ? 0.f : exp2f(mw - Mh);
                        Lh += f[w] * sl[w * kMaxGroup + h];
                    }
                }
                const float inv = 1.f / Lh;
#pragma unroll
                for (int w = 0; w < NW; ++w) f[w] *= inv;
                const size_t head = (size_t)it.b * H + it.kvh * G + h;
                const size_t pi = head * prm.max_partitions + it.slot;
#pragma unroll
                for (int kk = 0; kk < kSlice / 8; ++kk) {
                    const int d = warp * kSlice + 8 * kk + 2 * qd;
                    const float* r0 = rb + h * S::kRedStride + d;
                    float v0 = f[0] * r0[0], v1 = f[0] * r0[1];
#pragma unroll
                    for (int w = 1; w < NW; ++w) {
                        if (w < nw) {
                            const float* rw = rb + (w * kMaxGroup + h) * S::kRedStride + d;
                            v0 += f[w] * rw[0];
                            v1 += f[w] * rw[1];
                        }
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
    }
    // copies issued ahead of an abort complete before the CTA exits
    for (uint32_t x = pos; x < issued; ++x) mbar_wait(bar0 + 8 * (x % NS), (x / NS) & 1, kDefaultWaitLimit);
    PA_PT_MARK(4);
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
template <int D, int NW, int NS, bool Flat>
cudaError_t launch_persistent_t(const PartitionParams& prm, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                                cudaStream_t stream) {
    const int smem = PersistentShape<D, NW, NS>::kSmemBytes + persistent_seq_cache_bytes(prm.num_seqs);
    // the attribute allows the largest table cache, so it is set once per device
    constexpr int kSmemMax = PersistentShape<D, NW, NS>::kSmemBytes + persistent_seq_cache_bytes(kPersistentSeqCache);
    static_assert(kSmemMax <= 227 * 1024, "shared memory budget of one CTA with the table cache");
    static std::atomic<unsigned long long> done{0};
    cudaError_t e = once_per_device(done, [] {
        cudaError_t r = cudaFuncSetAttribute(pa_partition_persistent_kernel<D, NW, NS, Flat>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
        if (r != cudaSuccess) return r;
        // all of an SM's shared memory, so that the dependent reduce CTAs fit beside these
        return cudaFuncSetAttribute(pa_partition_persistent_kernel<D, NW, NS, Flat>,
                                    cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, pa_partition_persistent_kernel<D, NW, NS, Flat>, tk, tv, prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_partition_persistent(int head_dim, int warps, int stages, const PartitionParams& prm,
                                        const CUtensorMap& tk, const CUtensorMap& tv, int grid, cudaStream_t stream) {
    // the flat split needs no work list, but its tables must fit the CTA's cache
    const bool flat = prm.flat != 0;
    if (flat ? (prm.num_seqs > kPersistentSeqCache || prm.max_partitions < 1)
             : (!prm.work_offsets || !prm.work_counter || !prm.seq_order || !prm.part_sizes))
        return cudaErrorInvalidValue;
    if (grid <= 0) return cudaErrorInvalidValue;
#define PA_PLAUNCH_CASE(W_, S_)                                                                       \
    if (warps == W_ && stages == S_) {                                                               \
        switch (head_dim) {                                                                          \
            case 64:                                                                                 \
                return flat ? launch_persistent_t<64, W_, S_, true>(prm, tk, tv, grid, stream)        \
                            : launch_persistent_t<64, W_, S_, false>(prm, tk, tv, grid, stream);      \
            case 128:                                                                                \
                return flat ? launch_persistent_t<128, W_, S_, true>(prm, tk, tv, grid, stream)       \
                            : launch_persistent_t<128, W_, S_, false>(prm, tk, tv, grid, stream);     \
            case 256:                                                                                \
                return flat ? launch_persistent_t<256, W_, S_, true>(prm, tk, tv, grid, stream)       \
                            : launch_persistent_t<256, W_, S_, false>(prm, tk, tv, grid, stream);     \
            default: return cudaErrorInvalidValue;                                                   \
        }                                                                                            \
    }
    PA_FOR_EACH_PERSISTENT_SHAPE(PA_PLAUNCH_CASE)
#undef PA_PLAUNCH_CASE
    return cudaErrorInvalidValue;
}

// The work list of the persistent schedule, built by one CTA of 1024 threads
// (thread x handles a contiguous run of sequences):
//  1. T = the valid non-empty sequences' blocks and their count (block
//     reductions), then the apportioning cap: each round the 32 warps count
//     the partitions of 32 candidate caps at once;
//  2. each sequence's partition size (balanced_partition with the cap, or
//     with the caller's size) and item count: one per
//     (partition, kv head), one per kv head for an empty sequence (its output
//     is zeroed), one for an invalid length (it is reported);
//  3. the schedule order: a counting sort of the sequences by partition
//     length in blocks, longest first (empty and invalid ones last), so the
//     items handed out last are the shortest; the order within a length is
//     whatever the atomics give, which changes only which CTA takes an item,
//     never a result;
//  4. the exclusive prefix sums of the item counts in that order, and the item
//     counter reset to the grid size.
constexpr int kScanThreads = 1024;
constexpr int kOrderKeys = 1024;  // partition lengths in blocks, the longest clamped
static_assert(kOrderKeys == kScanThreads, "one key per thread in the key scan");

__device__ __forceinline__ bool scan_valid(const ScanParams& prm, int L) {
    return L >= 0 && L <= prm.max_seq_len && L <= prm.max_blocks_per_seq * kBlockSize;
}

// Block-wide exclusive scan of one int per thread (kScanThreads threads).
__device__ __forceinline__ int scan_block_exclusive(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += u;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(kFull, w, off);
            if (lane >= off) w += u;
        }
        warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int excl = incl - v + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (total) *total = warp_sums[kScanThreads / 32 - 1];
    __syncthreads();  // warp_sums may be reused by the caller
    return excl;
}

__global__ void __launch_bounds__(kScanThreads) pa_work_scan_kernel(const ScanParams prm) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ int cursor[kOrderKeys];  // per key: count, then next rank
    __shared__ int warp_sums[kScanThreads / 32];
    __shared__ int s_nblk[kScanThreads];  // blocks of sequence b when B <= kScanThreads (0: empty or invalid)
    __shared__ int s_fits[kScanThreads / 32];
    __shared__ unsigned long long s_blocks;
    __shared__ int s_count;
    const int B = prm.num_seqs;
    const int per = (B + kScanThreads - 1) / kScanThreads;
    const int b0 = threadIdx.x * per, b1 = min(B, b0 + per);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int x = threadIdx.x; x < kOrderKeys; x += kScanThreads) cursor[x] = 0;
    if (threadIdx.x == 0) {
        s_blocks = 0;
        s_count = 0;
    }
    __syncthreads();
    auto blocks_at = [&](int b) {
        const int L = __ldg(prm.seq_lens + b);
        return (scan_valid(prm, L) && L > 0) ? (L + kBlockSize - 1) / kBlockSize : 0;
    };

    // 1. the valid non-empty sequences' blocks and their count
    unsigned long long mine = 0;
    int cnt = 0;
    for (int b = b0; b < b1; ++b) {
        const int nb = blocks_at(b);
        if (B <= kScanThreads) s_nblk[b] = nb;
        if (nb) {
            mine += (unsigned long long)nb;
            ++cnt;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        mine += __shfl_xor_sync(kFull, mine, off);
        cnt += __shfl_xor_sync(kFull, cnt, off);
    }
    if (lane == 0 && cnt) {
        atomicAdd(&s_blocks, mine);
        atomicAdd(&s_count, cnt);
    }
    __syncthreads();
    // The apportioning cap: the smallest S with sum_b ceil(blocks_b / S) <= slots
    // (the count only falls as S grows).  lo = ceil(T / slots) is a lower
    // bound; with fewer sequences than slots, hi = ceil(T / (slots - count))
    // fits, since each ceiling adds less than one.  Each round the 32 warps
    // count the partitions of 32 caps spread over [lo, hi] at once and keep
    // the stretch below the smallest cap that fits: the range shrinks 32-fold
    // a round, one or two rounds in practice.
    long long cap = 1;
    if (prm.partition_size <= 0 && s_count > 0) {
        const long long Tb = (long long)s_blocks;
        const int slots = prm.slots, nv = s_count;
        long long lo = (Tb + slots - 1) / slots, hi = lo;
        if (nv < slots) hi = (Tb + (slots - nv) - 1) / (slots - nv);
        while (lo < hi) {  // lo and hi are the same on every thread
            const long long c = lo + ((hi - lo) * warp) / 32;
            unsigned long long parts = 0;
            for (int b = lane; b < B; b += 32) {
                const int nb = B <= kScanThreads ? s_nblk[b] : blocks_at(b);
                parts += (unsigned long long)((nb + c - 1) / c);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) parts += __shfl_xor_sync(kFull, parts, off);
            if (lane == 0) s_fits[warp] = parts <= (unsigned long long)slots;
            __syncthreads();
            int first = 32;  // the smallest candidate that fits
            for (int w = 31; w >= 0; --w)
                if (s_fits[w]) first = w;
            const long long c_first = lo + ((hi - lo) * (first < 32 ? first : 31)) / 32;
            const long long c_before = first > 0 ? lo + ((hi - lo) * (first - 1)) / 32 : lo - 1;
            if (first == 32) {
                lo = c_first + 1;
            } else {
                hi = c_first;
                lo = c_before + 1;
            }
            __syncthreads();  // s_fits is written again next round
        }
        cap = lo;
    }

    // 2. partition sizes, item counts, sort keys (bucket 0 = the longest)
    auto key_of = [&](int L, int part) {
        if (!scan_valid(prm, L) || L == 0) return kOrderKeys - 1;
        return kOrderKeys - 1 - min(part / kBlockSize, kOrderKeys - 1);
    };
    const int pmax = prm.partition_size > 0 ? prm.partition_size : (int)min(cap * kBlockSize, (long long)1 << 30);
    for (int b = b0; b < b1; ++b) {
        const int L = __ldg(prm.seq_lens + b);
        int part = kBlockSize;
        if (scan_valid(prm, L) && L > 0) part = balanced_partition(L, pmax);
        prm.part_sizes[b] = part;
        atomicAdd(&cursor[key_of(L, part)], 1);
    }
    __syncthreads();

    // 3. the first rank of each key, then every sequence's rank
    const int first = scan_block_exclusive(cursor[threadIdx.x], warp_sums, nullptr);
    cursor[threadIdx.x] = first;
    __syncthreads();
    for (int b = b0; b < b1; ++b) {
        const int L = __ldg(prm.seq_lens + b);
        const int part = prm.part_sizes[b];
        const int rank = atomicAdd(&cursor[key_of(L, part)], 1);
        int items = 1;  // an invalid length: one item reports it
        if (scan_valid(prm, L)) items = L == 0 ? prm.num_kv_heads : ((L + part - 1) / part) * prm.num_kv_heads;
        prm.seq_order[rank] = b;
        prm.work_offsets[rank] = items;  // turned into prefix sums below
    }
    __syncthreads();  // the block's global writes are visible to all its threads

    // 4. exclusive prefix sums over the schedule order, in place
    int local = 0;
    for (int r = b0; r < b1; ++r) local += prm.work_offsets[r];
    int total = 0;
    int run = scan_block_exclusive(local, warp_sums, &total);
    for (int r = b0; r < b1; ++r) {
        const int it = prm.work_offsets[r];
        prm.work_offsets[r] = run;
        run += it;
    }
    if (threadIdx.x == 0) {
        prm.work_offsets[B] = total;
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

}  // namespace pa
