// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05 +
// TMEM), for GB300.  Included by pa_prefix.cu after pa_prefix_kernel.cuh.
//
// Same operation and inputs as pa_prefix_kernel (see pa_prefix_kernel.cuh).
// Mapping:
// * one CTA per (query tile, kv head, sequence); the tile is 128 rows of
//   (new token, GQA head) pairs = floor(128 / G) tokens.  Three roles in
//   separate warps, handing over only through mbarriers:
//   - warps 0-3 (softmax): thread t owns row t (= TMEM lane t); it turns its
//     score row into P (fp16) with the online-softmax update and rescales
//     its O row in TMEM when its max moves;
//   - warps 4-7 (loads): warp i copies block i of every K and V tile, in the
//     order the MMAs consume them, each into a ring slot as soon as the MMA
//     that read the slot's previous tile has completed; their lanes keep the
//     block-table entries of the current and the next 32 blocks in registers;
//   - warp 8 (MMA, one lane issues): S(j+1) = Q K(j+1)^T (M 128, N 64,
//     K = head_dim) into one of two TMEM score buffers, then
//     O += P(j) V(j) (M 128, N = head_dim, K 64) with P read from one of two
//     TMEM P buffers; so S(j+1) runs on the tensor cores while the rows work
//     on tile j;
// * keys are walked in tiles of 64 (4 blocks of 16: paged context blocks
//   through the block table, then the chunk's own blocks), K tiles in a
//   3-slot ring and V tiles in a 2-slot ring, all with the 128-byte swizzle:
//   a K block as one 16-row box per 64 head_dim columns (the S operand needs
//   the 64 keys of a tile contiguous per column chunk), a V block as a single
//   box laid out [chunk][16 rows][128 B] (one P.V MMA per block reads it);
// * every wait is bounded; a wait that gives up sets PA_DEV_TIMEOUT and an
//   abort flag the other roles poll, and the CTA drains its copies and MMAs,
//   frees its TMEM and exits without writing.

constexpr int kTcRows = 128;   // MMA M: rows of (token, head)
constexpr int kTcKeys = 64;    // keys per tile: MMA N of S, K of P.V
constexpr int kTcKSlots = 3;
constexpr int kTcVSlots = 2;
constexpr int kTcSoftmaxWarps = kTcRows / 32;
constexpr int kTcLoadWarps = kTcKeys / kBlockSize;   // one per block of a key tile
constexpr int kTcLoadWarp0 = kTcSoftmaxWarps;
constexpr int kTcMmaWarp = kTcLoadWarp0 + kTcLoadWarps;
constexpr int kTcThreads = (kTcMmaWarp + 1) * 32;

// mbarriers of one CTA, by index
enum : int {
    kTcBarKFull = 0,                          // K slot landed (one arrival per load warp + copy bytes)
    kTcBarKEmpty = kTcBarKFull + kTcKSlots,   // K slot read by its S MMA (commit)
    kTcBarVFull = kTcBarKEmpty + kTcKSlots,   // V slot landed (as K)
    kTcBarVEmpty = kTcBarVFull + kTcVSlots,   // V slot read by its P.V MMA (commit)
    kTcBarSDone = kTcBarVEmpty + kTcVSlots,   // score buffer b written (commit), 2
    kTcBarPReady = kTcBarSDone + 2,           // P buffer b written by all 4 row warps, 2
    kTcBarODone = kTcBarPReady + 2,           // a P.V completed (commit)
    kTcBarMDone = kTcBarODone + 1,            // every MMA of the CTA completed (final commit)
    kTcBars = kTcBarMDone + 1
};

template <int D>
struct PrefixTcShape {
    static constexpr int kChunks = D / 64;
    static constexpr int kQBytes = kTcRows * D * 2;
    static constexpr int kTileBytes = kTcKeys * D * 2;          // K or V of one key tile
    static constexpr int kChunkStride = kTcKeys * 128;          // one 64-column chunk of a K tile
    static constexpr int kBlockBytes = kBlockSize * D * 2;      // one block of a V tile: [chunk][16][128 B]
    static constexpr int kCtrlBytes = kTcBars * 8 + 16;         // barriers, TMEM address, abort flag
    static constexpr int kSmemNeed = 1024 + kQBytes + (kTcKSlots + kTcVSlots) * kTileBytes + kCtrlBytes;
    // at most two CTAs per SM, so that their TMEM allocations always fit in
    // the SM's 512 columns (an allocation never has to wait for another CTA)
    static constexpr int kSmemBytes = kSmemNeed > 80 * 1024 ? kSmemNeed : 80 * 1024;
    // O (D columns), two score buffers (64 each), two P buffers (32 each)
    static constexpr int kTmemCols = D + 2 * kTcKeys + kTcKeys <= 256 ? 256 : 512;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget of one CTA");
};

// tcgen05 shared-memory matrix descriptor: 128-byte swizzle, given start,
// leading- and stride-dimension byte offsets (fixed version field 1).
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp16 A and B, fp32 accumulator.
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N, int b_mn_major) {
    return (1u << 4) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                 "l"(a), "l"(b), "r"(id), "r"(acc));
}

__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
                 "r"(a), "l"(b), "r"(id), "r"(acc));
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define PA_TC_REGS32(v)                                                                                          \
    "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),  \
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),   \
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),  \
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
#define PA_TC_IN32(v)                                                                                            \
    "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), \
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),         \
        "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]),          \
        "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])

// 32 consecutive 32-bit columns of this thread's TMEM lane, loaded and waited
// for in one statement: the destination registers of tcgen05.ld hold their
// values only after tcgen05.wait::ld, so no use may be scheduled in between.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : PA_TC_REGS32(v)
        : "r"(taddr)
        : "memory");
}

// The matching store, also waited for in the same statement: tcgen05.st reads
// its source registers until tcgen05.wait::st, so they must not be reused
// before it.
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        PA_TC_IN32(v)
        : "memory");
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, uint32_t limit, const volatile int* abort_flag) {
    for (uint32_t n = 0; n < limit; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63) == 63 && *abort_flag) return false;
    }
    return false;
}

__device__ __forceinline__ float tc_ex2(float x) {  // the PTX ex2.approx instruction, 2^x
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Diagnostic builds (-DPA_TRACE): SM clock stamps of pipeline events per key
// tile j, 16 slots: 0-3 and 12-13 by the MMA warp (loop top, S(j+1) issued,
// P(j) ready, V(j) landed, K(j+1) landed, P.V(j) issued), 4 and 8-11 by the
// load warp (V(j) issued, loop top, K(j+1) slot free, K(j+1) issued, V(j)
// slot free), 5-6 by warp 0 (scores j in, P(j) out) and 7 by warp 3 (P(j) out).
#ifdef PA_TRACE
#define PA_TC_MARK(j, e)                                                                                          \
    do {                                                                                                          \
        if (prm.trace && (j) < kPrefixTraceIters) {                                                               \
            const size_t cta_ = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;           \
            prm.trace[(cta_ * kPrefixTraceIters + (j)) * 16 + (e)] = (unsigned long long)clock64();              \
        }                                                                                                         \
    } while (0)
#else
#define PA_TC_MARK(j, e) \
    do {                 \
    } while (0)
#endif

// Block-table entries of one copy stream, held by the 32 lanes of a warp:
// lane l has the entry of block 32 g + l (g = the current group) and of
// block 32 (g + 1) + l, loaded one group ahead so the lookup latency is hidden.
struct TcBlockCursor {
    int group = -1;
    int cur = -1;
    int nxt = -1;
};

// Bounded wait by every lane of a warp; true only if all lanes saw the phase.
__device__ __forceinline__ bool tc_warp_wait(uint32_t bar, uint32_t parity, uint32_t limit,
                                             const volatile int* abort_flag) {
    const bool ok = tc_wait(bar, parity, limit, abort_flag);
    return __all_sync(kFull, ok);
}

__device__ __forceinline__ void tc_tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                               uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
        ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}

// AND of `ok` over the load warps (named barrier 1); every thread of those
// warps calls it at the same point, so they all take the same decision.
__device__ __forceinline__ bool tc_load_warps_agree(bool ok) {
    int r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.b32 pi, %1, 0;\n\tbar.red.and.pred po, 1, %2, pi;\n\t"
        "selp.s32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(ok ? 1 : 0), "r"(kTcLoadWarps * 32)
        : "memory");
    return r != 0;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    pa_prefix_tc_kernel(const __grid_constant__ CUtensorMap tmap_kc, const __grid_constant__ CUtensorMap tmap_vc,
                        const __grid_constant__ CUtensorMap tmap_kn, const __grid_constant__ CUtensorMap tmap_vn,
                        const PrefixParams prm) {
    using S = PrefixTcShape<D>;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* qs = smem;
    uint8_t* ks = qs + S::kQBytes;
    uint8_t* vs = ks + kTcKSlots * S::kTileBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(vs + kTcVSlots * S::kTileBytes);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kTcBars);
    volatile int* sm_abort = reinterpret_cast<volatile int*>(tslot + 1);
    const uint32_t bar0 = smem_addr(bars);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    const int tile = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int G = prm.group, H = prm.num_heads;
    const int tile_tokens = kTcRows / G;

    const int C = __ldg(prm.context_lens + b);
    const int q0 = __ldg(prm.query_start_loc + b), q1 = __ldg(prm.query_start_loc + b + 1);
    const int qlen = q1 - q0;
    if (C < 0 || C > prm.max_context_len || C > prm.max_blocks_per_seq * kBlockSize || qlen < 0 ||
        qlen > prm.max_query_len || q0 < 0 || q1 > prm.num_tokens) {
        if (tile == 0 && kvh == 0 && t == 0) atomicOr(prm.status, PA_DEV_BAD_SEQ_LEN);
        return;
    }
    const int t0 = tile * tile_tokens;
    if (t0 >= qlen) return;
    const int tlast = min(qlen, t0 + tile_tokens) - 1;
    const int nctx = (C + kBlockSize - 1) / kBlockSize;         // context blocks
    const int nblocks = nctx + tlast / kBlockSize + 1;          // + chunk blocks up to tlast
    const int ntiles = (nblocks + 3) / 4;
    const int32_t* bt = prm.block_tables + (size_t)b * prm.max_blocks_per_seq;

    if (t == 0) {
        *sm_abort = 0;
        for (int i = 0; i < kTcBars; ++i)
            mbar_init(bar(i), (i == kTcBarPReady || i == kTcBarPReady + 1) ? kTcSoftmaxWarps
                              : (i < kTcBarKEmpty || (i >= kTcBarVFull && i < kTcBarVEmpty)) ? kTcLoadWarps
                                                                                           : 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tslot)),
                     "r"(S::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    // Q tile: row r = (token t0 + r / G, head kvh * G + r % G), 64-column
    // chunks of 128 rows x 128 B with the 128-byte swizzle; missing rows are 0.
    for (int idx = t; idx < kTcRows * (D / 8); idx += kTcThreads) {
        const int r = idx / (D / 8), u = idx % (D / 8);
        const int ti = r / G, h = r % G;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (ti < tile_tokens && t0 + ti < qlen)
            v = __ldg(reinterpret_cast<const uint4*>(prm.q + ((size_t)(q0 + t0 + ti) * H + kvh * G + h) * D) + u);
        *reinterpret_cast<uint4*>(qs + (u >> 3) * (kTcRows * 128) + r * 128 + (((u & 7) ^ (r & 7)) << 4)) = v;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tO = tmem;                    // D columns
    const uint32_t tS0 = tmem + D;               // two score buffers of 64 columns
    const uint32_t tP0 = tS0 + 2 * kTcKeys;      // two P buffers of 32 columns (fp16 pairs)
    const unsigned limit = prm.force_timeout ? 0u : prm.wait_limit;

    if (warp >= kTcLoadWarp0 && warp < kTcMmaWarp) {
        // ---------------- load warps: warp i copies block i of every key tile ----------------
        // Copies go in the order the MMAs use them (S(0), S(1), P.V(0), S(2),
        // P.V(1), ...: K(j+1) before V(j)).  A TMA instruction occupies its
        // issuing thread for a fixed time whatever the box size, so four warps
        // issue in parallel; they agree on every wait so that a tile is copied
        // by all four or by none.
        const int i = warp - kTcLoadWarp0;
        TcBlockCursor kcur, vcur;
        auto fetch = [&](int g) {
            const int blk = 32 * g + lane;
            return blk < nctx ? __ldg(bt + blk) : -1;
        };
        // physical block of block blk of the sequence (meaningful for blk < nctx); warp-collective
        auto lookup = [&](TcBlockCursor& c, int blk) {
            const int g = blk >> 5;
            if (g != c.group) {
                c.cur = g == c.group + 1 ? c.nxt : fetch(g);
                c.nxt = fetch(g + 1);
                c.group = g;
            }
            return __shfl_sync(kFull, c.cur, blk & 31);
        };
        // block blk of a tile: context block blk when below nctx (-2 for an
        // invalid id: read zeros instead), else chunk block blk - nctx (-1)
        auto checked = [&](int blk, int phys) {
            if (blk >= nctx) return -1;
            if (phys < 0 || (long long)phys >= prm.num_blocks) {
                atomicOr(prm.status, PA_DEV_BAD_BLOCK_ID);
                return -2;
            }
            return phys;
        };
        auto chunk_token = [&](int blk, int p) { return p == -2 ? prm.num_tokens : q0 + (blk - nctx) * kBlockSize; };
        // K: head_dim/64 boxes of 16 rows x 64 columns, into rows 16 i.. of
        // every 64-column chunk of the slot (the S MMA's operand layout)
        auto issue_k = [&](int j) {
            const int blk = 4 * j + i;
            const int phys = lookup(kcur, blk);
            if (lane == 0) {
                const uint32_t full = bar(kTcBarKFull + j % kTcKSlots);
                const uint32_t dst = smem_addr(ks + (j % kTcKSlots) * S::kTileBytes) + i * (kBlockSize * 128);
                mbar_arrive_expect_tx(full, S::kBlockBytes);
                const int p = checked(blk, phys);
#pragma unroll
                for (int ch = 0; ch < S::kChunks; ++ch) {
                    if (p >= 0)
                        tma_load_2d(dst + ch * S::kChunkStride, &tmap_kc, ch * 64,
                                    (p * prm.num_kv_heads + kvh) * kBlockSize, full);
                    else
                        tma_load_3d(dst + ch * S::kChunkStride, &tmap_kn, ch * 64, kvh, chunk_token(blk, p), full);
                }
            }
            __syncwarp();
        };
        // V: the whole block in one box, [chunk][16 rows][128 B], block i of the slot
        auto issue_v = [&](int j) {
            const int blk = 4 * j + i;
            const int phys = lookup(vcur, blk);
            if (lane == 0) {
                const uint32_t full = bar(kTcBarVFull + j % kTcVSlots);
                const uint32_t dst = smem_addr(vs + (j % kTcVSlots) * S::kTileBytes) + i * S::kBlockBytes;
                mbar_arrive_expect_tx(full, S::kBlockBytes);
                const int p = checked(blk, phys);
                if (p >= 0)
                    tma_load_3d(dst, &tmap_vc, 0, (p * prm.num_kv_heads + kvh) * kBlockSize, 0, full);
                else
                    tc_tma_load_4d(dst, &tmap_vn, 0, kvh, chunk_token(blk, p), 0, full);
            }
            __syncwarp();
        };
        kcur.nxt = vcur.nxt = fetch(0);
        bool ok = true;
        int k_issued = 0, v_issued = 0;
        if (ntiles > 0) {
            issue_k(0);
            k_issued = 1;
        }
        for (int j = 0; j < ntiles; ++j) {
            const int kj = j + 1;
            if (lane == 0 && i == 0) PA_TC_MARK(j, 8);
            if (kj < ntiles) {
                // slot kj % 3 last held K(kj - 3): free once S(kj - 3) has completed
                if (kj >= kTcKSlots &&
                    !(ok = tc_load_warps_agree(tc_warp_wait(bar(kTcBarKEmpty + kj % kTcKSlots),
                                                            (kj / kTcKSlots - 1) & 1, limit, sm_abort))))
                    break;
                if (lane == 0 && i == 0) PA_TC_MARK(j, 9);
                issue_k(kj);
                k_issued = kj + 1;
            }
            if (lane == 0 && i == 0) PA_TC_MARK(j, 10);
            // slot j % 2 last held V(j - 2): free once P.V(j - 2) has completed
            if (j >= kTcVSlots &&
                !(ok = tc_load_warps_agree(tc_warp_wait(bar(kTcBarVEmpty + j % kTcVSlots), (j / kTcVSlots - 1) & 1,
                                                        limit, sm_abort))))
                break;
            if (lane == 0 && i == 0) PA_TC_MARK(j, 11);
            issue_v(j);
            v_issued = j + 1;
            if (lane == 0 && i == 0) PA_TC_MARK(j, 4);
        }
        if (lane == 0) {
            if (!ok && i == 0) {
                *sm_abort = 1;
                atomicOr(prm.status, PA_DEV_TIMEOUT);
            }
            // every copy issued lands before the CTA exits: all four warps
            // issued the same tiles, and a slot holds at most one copy that
            // nobody may have waited for (the latest one)
            for (int x = max(0, k_issued - kTcKSlots); x < k_issued; ++x)
                mbar_wait(bar(kTcBarKFull + x % kTcKSlots), (x / kTcKSlots) & 1, kDefaultWaitLimit);
            for (int x = max(0, v_issued - kTcVSlots); x < v_issued; ++x)
                mbar_wait(bar(kTcBarVFull + x % kTcVSlots), (x / kTcVSlots) & 1, kDefaultWaitLimit);
        }
        __syncwarp();
    } else if (warp == kTcMmaWarp) {
        // ---------------- MMA warp: lane 0 issues, every lane waits ----------------
        constexpr uint32_t idS = tc_idesc(kTcRows, kTcKeys, 0);
        constexpr uint32_t idO = tc_idesc(kTcRows, D, 1);
        const uint32_t qb = smem_addr(qs);
        const int partial_tile = C % kBlockSize != 0 ? (nctx - 1) / 4 : -1;
        // S(j) = Q K(j)^T into score buffer j % 2; K slot j % 3 is free when it completes
        auto issue_s = [&](int j) {
            if (lane == 0) {
                const uint32_t kb = smem_addr(ks + (j % kTcKSlots) * S::kTileBytes);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t qo = (k >> 2) * (kTcRows * 128) + (k & 3) * 32;
                    const uint32_t ko = (k >> 2) * S::kChunkStride + (k & 3) * 32;
                    tc_mma_ss(tS0 + (j & 1) * kTcKeys, tc_desc(qb + qo, 16, 1024), tc_desc(kb + ko, 16, 1024), idS,
                              k > 0);
                }
                tc_commit(bar(kTcBarSDone + (j & 1)));
                tc_commit(bar(kTcBarKEmpty + j % kTcKSlots));
            }
            __syncwarp();
        };
        bool ok = tc_warp_wait(bar(kTcBarKFull), 0, limit, sm_abort);
        if (ok) {
            tc_fence_after();
            issue_s(0);
        }
        for (int j = 0; ok && j < ntiles; ++j) {
            if (lane == 0) PA_TC_MARK(j, 0);
            if (j + 1 < ntiles) {
                // score buffer (j+1) % 2 last held S(j-1); the rows read it
                // before P(j-1) was ready, which the previous step waited for
                if (!(ok = tc_warp_wait(bar(kTcBarKFull + (j + 1) % kTcKSlots), ((j + 1) / kTcKSlots) & 1, limit,
                                        sm_abort)))
                    break;
                if (lane == 0) PA_TC_MARK(j, 12);
                tc_fence_after();
                issue_s(j + 1);
            }
            if (lane == 0) PA_TC_MARK(j, 1);
            // rows have written P(j) (and rescaled O if they had to)
            if (!(ok = tc_warp_wait(bar(kTcBarPReady + (j & 1)), (j >> 1) & 1, limit, sm_abort))) break;
            if (lane == 0) PA_TC_MARK(j, 2);
            if (!(ok = tc_warp_wait(bar(kTcBarVFull + j % kTcVSlots), (j / kTcVSlots) & 1, limit, sm_abort))) break;
            if (lane == 0) PA_TC_MARK(j, 3);
            uint8_t* vt = vs + (j % kTcVSlots) * S::kTileBytes;
            if (j == partial_tile) {
                // V rows of cache slots past the context may hold anything: p is
                // 0 there, but 0 * NaN is not; clear them before P.V reads them
                const int i = (nctx - 1) % 4, first = C % kBlockSize;
                const int units = (kBlockSize - first) * S::kChunks * 8;
                uint8_t* vb = vt + i * S::kBlockBytes;
                for (int x = lane; x < units; x += 32) {
                    const int r = first + x / (S::kChunks * 8), u = x % (S::kChunks * 8);
                    *reinterpret_cast<uint4*>(vb + (u >> 3) * (kBlockSize * 128) + r * 128 + (u & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
                // O += P(j) V(j), P in buffer j % 2, one MMA per block of 16 keys
                // (V block: 64-column chunks 2 KB apart, 8-key groups 1 KB
                // apart); V slot j % 2 is free when they complete
                const uint32_t vb = smem_addr(vt);
#pragma unroll
                for (int k = 0; k < kTcKeys / 16; ++k)
                    tc_mma_ts(tO, tP0 + (j & 1) * (kTcKeys / 2) + k * 8,
                              tc_desc(vb + k * S::kBlockBytes, kBlockSize * 128, 1024), idO, (j > 0 || k > 0));
                tc_commit(bar(kTcBarODone));
                tc_commit(bar(kTcBarVEmpty + j % kTcVSlots));
                PA_TC_MARK(j, 13);
            }
            __syncwarp();
        }
        if (lane == 0) {
            if (!ok) {
                *sm_abort = 1;
                atomicOr(prm.status, PA_DEV_TIMEOUT);
            }
            // every MMA issued above has completed once this commit arrives
            tc_commit(bar(kTcBarMDone));
            mbar_wait(bar(kTcBarMDone), 0, kDefaultWaitLimit);
        }
        __syncwarp();
    } else {
        // ---------------- softmax warps: thread t owns row t (TMEM lane t) ----------------
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const int ti = t / G;
        const int my_tok = t0 + ti;  // chunk token index of the row
        const bool row_real = ti < tile_tokens && my_tok < qlen;
        const float sl2 = prm.scale_log2;
        const uint32_t odone = bar(kTcBarODone);
        float m = -INFINITY, l = 0.f;  // reference max (scaled, log2 domain) and exp sum
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            if (!(ok = tc_warp_wait(bar(kTcBarSDone + (j & 1)), (j >> 1) & 1, limit, sm_abort))) break;
            tc_fence_after();
            if (t == 0) PA_TC_MARK(j, 5);
            uint32_t sv[2][32];
            const uint32_t tS = tS0 + (j & 1) * kTcKeys + lane_off;
            tc_ld32(tS, sv[0]);
            tc_ld32(tS + 32, sv[1]);
            // visibility: every key of a tile made only of full context blocks
            // is visible; otherwise mask per key
            const bool full_ctx = 4 * j + 3 < nctx - (C % kBlockSize != 0 ? 1 : 0);
            if (!full_ctx) {
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int col = h2 * 32 + c;
                        const int blk = 4 * j + (col >> 4), slot = col & 15;
                        const bool vis = blk < nctx ? blk * kBlockSize + slot < C
                                                    : ((blk - nctx) * kBlockSize + slot <= my_tok);
                        if (!vis) sv[h2][c] = __float_as_uint(sl2 >= 0.f ? -INFINITY : INFINITY);
                    }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
            for (int c = 0; c < 32; c += 2) {  // on scaled scores: the scale may be negative
                mx0 = fmaxf(mx0, __uint_as_float(sv[0][c]) * sl2);
                mx1 = fmaxf(mx1, __uint_as_float(sv[0][c + 1]) * sl2);
                mx2 = fmaxf(mx2, __uint_as_float(sv[1][c]) * sl2);
                mx3 = fmaxf(mx3, __uint_as_float(sv[1][c + 1]) * sl2);
            }
            const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
            // The reference max m only moves when the tile max exceeds it by
            // more than 2^8 (then O and l are rescaled); otherwise p = 2^(s - m)
            // <= 2^8 is exact enough in fp16 and O stays untouched.
            const bool move = mx > m + 8.f;  // also true on the first visible tile (m = -inf)
            const float mref = move ? mx : m;
            const float base = mref == -INFINITY ? 0.f : mref;
            const float alpha = move ? tc_ex2(m - base) : 1.f;
            m = mref;
            uint32_t pk[32];
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const int h2 = c >> 4, cc = (c & 15) * 2;
                const float p0 = tc_ex2(fmaf(__uint_as_float(sv[h2][cc]), sl2, -base));
                const float p1 = tc_ex2(fmaf(__uint_as_float(sv[h2][cc + 1]), sl2, -base));
                rs0 += p0;
                rs1 += p1;
                pk[c] = half2_bits(__floats2half2_rn(p0, p1));
            }
            l = l * alpha + (rs0 + rs1);
            // P(j) to its own buffer; P.V(j-2), its last reader, was issued
            // before S(j) and so completed before S(j) did
            tc_st32(tP0 + (j & 1) * (kTcKeys / 2) + lane_off, pk);
            if (j > 0 && __any_sync(kFull, move)) {
                // O is written by P.V(j-1): wait for it, then rescale this row.
                // P.V(j-2) completed before S(j), so odone is at most one phase
                // behind and the parity wait is unambiguous.
                if (!(ok = tc_warp_wait(odone, (j - 1) & 1, limit, sm_abort))) break;
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t ov[32];
                    tc_ld32(tO + lane_off + c0, ov);
#pragma unroll
                    for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
                    tc_st32(tO + lane_off + c0, ov);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (t == 0) PA_TC_MARK(j, 6);
            if (t == 96) PA_TC_MARK(j, 7);
            if (lane == 0) mbar_arrive(bar(kTcBarPReady + (j & 1)));
        }
        // odone completes once per P.V, in issue order.  S(ntiles-1) was issued
        // before P.V(ntiles-2), so that P.V may still run here; a parity wait
        // only tells phases apart within one of the current phase, so wait
        // for phase ntiles-2 before phase ntiles-1.
        if (ok && ntiles >= 2) ok = tc_warp_wait(odone, (ntiles - 2) & 1, limit, sm_abort);
        if (ok) ok = tc_warp_wait(odone, (ntiles - 1) & 1, limit, sm_abort);
        if (!ok) {
            if (lane == 0) {
                *sm_abort = 1;
                atomicOr(prm.status, PA_DEV_TIMEOUT);
            }
        } else {
            tc_fence_after();
            // O / l to fp16 for the rows that exist
            const float inv = 1.f / l;
            __half* orow = prm.out + ((size_t)(q0 + my_tok) * H + kvh * G + (t % G)) * D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t ov[32];
                tc_ld32(tO + lane_off + c0, ov);
                if (row_real) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 w;
                        uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            wp[e] = half2_bits(__floats2half2_rn(__uint_as_float(ov[c + 2 * e]) * inv,
                                                                 __uint_as_float(ov[c + 2 * e + 1]) * inv));
                        *reinterpret_cast<uint4*>(orow + c0 + c) = w;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();  // every role done: no copy or MMA in flight past this point
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(S::kTmemCols));
}

int prefix_tc_smem_bytes(int head_dim) {
    switch (head_dim) {
        case 64: return PrefixTcShape<64>::kSmemBytes;
        case 128: return PrefixTcShape<128>::kSmemBytes;
        case 256: return PrefixTcShape<256>::kSmemBytes;
        default: return -1;
    }
}

namespace {
template <int D>
cudaError_t launch_prefix_tc_t(const PrefixParams& prm, const CUtensorMap* maps, dim3 grid, cudaStream_t stream) {
    const int smem = PrefixTcShape<D>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(pa_prefix_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, pa_prefix_tc_kernel<D>, maps[0], maps[1], maps[2], maps[3], prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_prefix_tc(int head_dim, const PrefixParams& prm, const CUtensorMap* maps, dim3 grid,
                             cudaStream_t stream) {
    switch (head_dim) {
        case 64: return launch_prefix_tc_t<64>(prm, maps, grid, stream);
        case 128: return launch_prefix_tc_t<128>(prm, maps, grid, stream);
        case 256: return launch_prefix_tc_t<256>(prm, maps, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}
