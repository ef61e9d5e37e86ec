// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05 +
// TMEM), for GB300.  Included by pa_prefix.cu after pa_prefix_kernel.cuh.
//
// Same operation and inputs as pa_prefix_kernel (see pa_prefix_kernel.cuh).
// Mapping:
// * a unit of work is a (query tile, kv head, sequence); the tile is 128 rows
//   of (new token, GQA head) pairs = floor(128 / G) tokens.  By default a grid
//   of the CTAs the SMs hold at once claims the units from a device counter
//   (the persistent form; the grid form runs one CTA per unit), and each CTA's
//   rings and barrier phases run on from one unit to the next.  Three roles
//   in separate warps, handing over only through mbarriers:
//   - warps 0-3 (softmax): thread t owns row t (= TMEM lane t); it turns its
//     score row into P (fp16) with the online-softmax update and rescales
//     its O row in TMEM when its max moves;
//   - warps 4-13 (loads): eight copy K (two per block of a tile), two copy V
//     (two blocks each), each group into its ring slot as soon as the MMA that
//     read the slot's previous tile has completed; their lanes keep the
//     block-table entries of the current and the next 32 blocks in registers;
//   - warps 14 and 15 (MMA, one lane each): warp 14 issues S(j) = Q K(j)^T
//     (M 128, N 64, K = head_dim, Q read from TMEM so only K comes from
//     shared memory) into TMEM score buffer j % 2 as soon as the P.V that
//     last read that buffer has completed, warp 15 O += P(j) V(j) (M 128,
//     N = head_dim, K 64) with P(j) read from the same buffer, where the rows
//     wrote it (fp16) over S(j).  The tensor cores take few MMAs ahead of
//     their issuer, so two issuing threads keep them busy while either waits;
//     with two score buffers S(j+1) is issued right behind S(j) and runs
//     while the rows work on tile j, with no hand-over from the rows first;
// * keys are walked in tiles of 64 (4 blocks of 16: paged context blocks
//   through the block table, then the chunk's own blocks), K tiles in a
//   4-slot ring and V tiles in a 3-slot ring (4 below head_dim 256), all with
//   the 128-byte swizzle:
//   a K block as one 16-row box per 64 head_dim columns (the S operand needs
//   the 64 keys of a tile contiguous per column chunk), a V block as a single
//   box laid out [chunk][16 rows][128 B] (one P.V MMA per block reads it);
// * every wait is bounded; a wait that gives up sets PA_DEV_TIMEOUT and an
//   abort flag the other roles poll, and the CTA drains its copies and MMAs,
//   frees its TMEM and exits without writing.

constexpr int kTcRows = 128;   // MMA M: rows of (token, head)
constexpr int kTcKeys = 64;    // keys per tile: MMA N of S, K of P.V
constexpr int kTcMaxSlots = 4;  // K or V ring slots at most
constexpr int kTcClaimAhead = 4;  // key tiles before a unit's end at which the next unit is claimed
constexpr int kTcSoftmaxWarps = kTcRows / 32;
constexpr int kTcKLoadWarps = 2 * (kTcKeys / kBlockSize);  // two per K block of a key tile
constexpr int kTcVLoadWarps = 2;                           // each copies every other V block
constexpr int kTcLoadWarps = kTcKLoadWarps + kTcVLoadWarps;
constexpr int kTcLoadWarp0 = kTcSoftmaxWarps;
constexpr int kTcSWarp = kTcLoadWarp0 + kTcLoadWarps;  // issues the S MMAs
constexpr int kTcPVWarp = kTcSWarp + 1;                // issues the P.V MMAs
constexpr int kTcThreads = (kTcPVWarp + 1) * 32;
// registers per thread: the SM's 64 K registers over the CTA's threads, in
// the allocation unit of 8
constexpr int kTcMaxRegs = (65536 / kTcThreads) / 8 * 8;

// mbarriers of one CTA, by index
enum : int {
    kTcBarKFull = 0,                          // K slot landed (one arrival per load warp + copy bytes)
    kTcBarKEmpty = kTcBarKFull + kTcMaxSlots,   // K slot read by its S MMA (commit)
    kTcBarVFull = kTcBarKEmpty + kTcMaxSlots,   // V slot landed (as K)
    kTcBarVEmpty = kTcBarVFull + kTcMaxSlots,   // V slot read by its P.V MMA (commit)
    kTcBarSDone = kTcBarVEmpty + kTcMaxSlots,   // score buffer b holds S(j) (commit), 2
    kTcBarPReady = kTcBarSDone + 2,           // P(j) written over S(j) in buffer b by all 4 row warps, 2
    kTcBarPVDone = kTcBarPReady + 2,          // the P.V reading buffer b completed (commit), 2
    kTcBarQReady = kTcBarPVDone + 2,          // Q rows stored in TMEM by the 4 row warps
    kTcBarSDrain = kTcBarQReady + 1,          // every S MMA completed (final commit)
    kTcBarPVDrain = kTcBarSDrain + 1,         // every P.V MMA completed (final commit)
    kTcBarQFree = kTcBarPVDrain + 1,          // a unit's S MMAs completed: Q may be rewritten (commit)
    kTcBarUnitFull = kTcBarQFree + 1,         // persistent form: unit id slot u % 2 written (claimer), 2
    kTcBarUnitEmpty = kTcBarUnitFull + 2,     // unit id slot u % 2 read by every warp, 2
    kTcBars = kTcBarUnitEmpty + 2
};

template <int D>
struct PrefixTcShape {
    static constexpr int kChunks = D / 64;
    static constexpr int kTileBytes = kTcKeys * D * 2;          // K or V of one key tile
    static constexpr int kChunkStride = kTcKeys * 128;          // one 64-column chunk of a K tile
    static constexpr int kBlockBytes = kBlockSize * D * 2;      // one block of a V tile: [chunk][16][128 B]
    // barriers, TMEM address, abort flag, 2 unit ids, 2 decoded units, the
    // row warps' copies of their current unit
    static constexpr int kCtrlBytes = kTcBars * 8 + 16 + 128 + 4 * 64;
    // ring slots: 7 tiles of 32 KB fill the shared memory at head_dim 256
    static constexpr int kKSlots = 4;
    static constexpr int kVSlots = D == 256 ? 3 : 4;
    static constexpr int kSmemNeed = 1024 + (kKSlots + kVSlots) * kTileBytes + kCtrlBytes;
    // at most two CTAs per SM, so that their TMEM allocations always fit in
    // the SM's 512 columns (an allocation never has to wait for another CTA)
    static constexpr int kSmemBytes = kSmemNeed > 80 * 1024 ? kSmemNeed : 80 * 1024;
    // O (D columns), Q (D / 2 columns of fp16 pairs), two score buffers of
    // 64 columns (each also takes its tile's P, 32 columns of fp16 pairs)
    static constexpr int kTmemUsed = D + D / 2 + 2 * kTcKeys;
    static constexpr int kTmemCols = kTmemUsed <= 256 ? 256 : 512;
    static_assert(kTmemUsed <= 512, "tensor memory columns of one SM");
    static_assert(kKSlots <= kTcMaxSlots && kVSlots <= kTcMaxSlots, "ring barriers");
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

// Two such loads (64 columns, e.g. two 32-column chunks) in flight under one
// wait::ld.
__device__ __forceinline__ void tc_ld32x2(uint32_t taddr0, uint32_t (&v)[32], uint32_t taddr1, uint32_t (&w)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : PA_TC_REGS32(v), PA_TC_REGS32(w)
        : "r"(taddr0), "r"(taddr1)
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

// Two such stores (two 32-column chunks) under one wait::st.
__device__ __forceinline__ void tc_st32x2(uint32_t taddr0, const uint32_t (&v)[32], uint32_t taddr1,
                                          const uint32_t (&w)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};\n\t"
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%1], {%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
        "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr0),
        "r"(taddr1), PA_TC_IN32(v), PA_TC_IN32(w)
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
// tile j (counted over all the CTA's units), 16 slots: 0-3 and 12-13 by the MMA warp (loop top, S(j+1) issued,
// P(j) ready, V(j) landed, K(j+1) landed, P.V(j) issued), 4 and 8-11 by the
// load warp (V(j) issued, loop top, K(j+1) slot free, K(j+1) issued, V(j)
// slot free), 5-6 by warp 0 (scores j in, P(j) out), 7 by warp 3 (P(j) out),
// 14-15 by the S warp (K(j) landed, score buffer j % 2 free).
#ifdef PA_TRACE
#define PA_TC_MARK(j, e)                                                                                          \
    do {                                                                                                          \
        if (prm.trace && (j) < kPrefixTraceIters - 1) {                                                           \
            const size_t cta_ = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;           \
            prm.trace[(cta_ * kPrefixTraceIters + (j)) * 16 + (e)] = (unsigned long long)clock64();              \
        }                                                                                                         \
    } while (0)
// Per-CTA phases in global-timer ns, in the last record of the CTA: 0 entry,
// 1 setup done, 2 Q in tensor memory (row thread 0), 3 tile loop done, 4 O
// stored, 5 every role done, 7 the SM id; at the persistent form's last
// switch between units (row thread 0): 8 tile loop done, 9 next unit read,
// 10 Q free, 11 next Q in tensor memory, 12 last P.Vs done, 13 O stored.
#define PA_TC_PHASE(e)                                                                                            \
    do {                                                                                                          \
        if (prm.trace && threadIdx.x == 0) {                                                                      \
            const size_t cta_ = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;           \
            unsigned long long g_;                                                                                \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g_));                                               \
            prm.trace[(cta_ * kPrefixTraceIters + kPrefixTraceIters - 1) * 16 + (e)] = (e) == 7 ? smid_of() : g_; \
        }                                                                                                         \
    } while (0)
__device__ __forceinline__ unsigned long long smid_of() {
    unsigned s;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
    return s;
}
#else
#define PA_TC_MARK(j, e) \
    do {                 \
    } while (0)
#define PA_TC_PHASE(e) \
    do {               \
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

// AND of `ok` over a group of warps (named barrier `id`, `threads` threads);
// every thread of the group calls it at the same point, so they all take the
// same decision.
__device__ __forceinline__ bool tc_group_agree(bool ok, int id, int threads) {
    int r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.b32 pi, %1, 0;\n\tbar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.s32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(ok ? 1 : 0), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

// A unit of the kernel's work: a query tile of one (sequence, kv head),
// whole or, in a key split (PrefixParams::split_parts), part `part` of its key
// tiles.  Units are numbered as the CTAs of the split's 1-D grid: the whole
// tiles first (tile fastest, then kv head, then sequence), then split_parts
// parts of each remaining tile.  Every role decodes the units it walks itself,
// from the same number, so they agree without a hand-over.
struct TcUnit {
    int b, kvh, tile, part, unit_r;
    int C, q0, qlen, t0;  // context length, first new token, new tokens, first token of the tile
    int nctx, jb, n;      // context blocks; key tiles [jb, jb + n) of the walk
    bool run;             // false: nothing to compute (a tile past the new tokens, or bad lengths)
};

__device__ __forceinline__ TcUnit tc_unit(const PrefixParams& prm, int c, bool report) {
    TcUnit u;
    int w = c;
    u.part = -1;
    u.unit_r = 0;
    if (prm.split_parts > 0 && c >= prm.split_whole) {
        u.unit_r = (c - prm.split_whole) / prm.split_parts;
        u.part = (c - prm.split_whole) - u.unit_r * prm.split_parts;
        w = prm.split_whole + u.unit_r;
    }
    u.tile = w % prm.tiles_per_seq;
    u.kvh = (w / prm.tiles_per_seq) % prm.num_kv_heads;
    u.b = w / (prm.tiles_per_seq * prm.num_kv_heads);
    u.C = __ldg(prm.context_lens + u.b);
    u.q0 = __ldg(prm.query_start_loc + u.b);
    u.qlen = __ldg(prm.query_start_loc + u.b + 1) - u.q0;
    u.t0 = u.tile * (kTcRows / prm.group);
    u.nctx = 0;
    u.jb = 0;
    u.n = 0;
    u.run = false;
    if (u.C < 0 || u.C > prm.max_context_len || u.C > prm.max_blocks_per_seq * kBlockSize || u.qlen < 0 ||
        u.qlen > prm.max_query_len || u.q0 < 0 || u.q0 + u.qlen > prm.num_tokens) {
        if (report && u.tile == 0 && u.kvh == 0) atomicOr(prm.status, PA_DEV_BAD_SEQ_LEN);
        return u;
    }
    if (u.t0 >= u.qlen) return u;
    const int tlast = min(u.qlen, u.t0 + kTcRows / prm.group) - 1;
    u.nctx = (u.C + kBlockSize - 1) / kBlockSize;         // context blocks
    const int nblocks = u.nctx + tlast / kBlockSize + 1;  // + chunk blocks up to tlast
    const int ntiles = (nblocks + 3) / 4;
    u.n = ntiles;
    if (u.part >= 0) {
        // part p walks [floor(p n / k), floor((p + 1) n / k)), in 32-bit terms
        // (n = q k + r: floor(p n / k) = p q + floor(p r / k)); a 64-bit
        // division here, a subroutine call inside the warp roles' branches,
        // made every role's tile loop about 20 % slower
        const int k = prm.split_parts, q = ntiles / k, r = ntiles - q * k;
        u.jb = u.part * q + (u.part * r) / k;
        u.n = (u.part + 1) * q + ((u.part + 1) * r) / k - u.jb;
    }
    u.run = true;
    return u;
}

template <int D, bool Persist>
__global__ void __maxnreg__(kTcMaxRegs)
    pa_prefix_tc_kernel(const __grid_constant__ CUtensorMap tmap_kc, const __grid_constant__ CUtensorMap tmap_vc,
                        const __grid_constant__ CUtensorMap tmap_kn, const __grid_constant__ CUtensorMap tmap_vn,
                        const PrefixParams prm) {
    using S = PrefixTcShape<D>;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* ks = smem;
    uint8_t* vs = ks + S::kKSlots * S::kTileBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(vs + S::kVSlots * S::kTileBytes);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kTcBars);
    volatile int* sm_abort = reinterpret_cast<volatile int*>(tslot + 1);
    volatile int* sm_unit = reinterpret_cast<volatile int*>(tslot + 2);  // 2 unit id slots
    TcUnit* sm_units = reinterpret_cast<TcUnit*>(tslot + 4);             // their decoded units
    TcUnit* rows_units = reinterpret_cast<TcUnit*>(reinterpret_cast<uint8_t*>(sm_units) + 128);  // one per row warp
    const uint32_t bar0 = smem_addr(bars);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const unsigned limit = prm.force_timeout ? 0u : prm.wait_limit;

    // Grid form: the CTA's one unit is its own (1-D grid of a key split, else
    // (query tiles, kv heads, sequences)).  Persistent form (prm.sched): a
    // fixed grid whose CTAs claim units from the device counter sched[0] in
    // number order until all are taken; the rings and barrier phases run on
    // across units, so a unit's first copies overlap the last one's MMAs and
    // epilogue, and the setup is paid once per CTA.
    // Persist: the persistent form (prm.sched set); its own instance, since
    // compiled apart from the grid form it measured 1 % faster at head_dim 128
    constexpr bool persist = Persist;
    const int c0 = prm.split_parts > 0 ? (int)blockIdx.x
                                       : (int)((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x);
    PA_TC_PHASE(0);
    PA_TC_PHASE(7);
    const int G = prm.group, H = prm.num_heads;
    TcUnit u0{};  // grid form: the CTA's unit
    if (!persist) {
        u0 = tc_unit(prm, c0, t == 0);
        if (!u0.run) return;
        // The row threads read their Q rows into registers after the setup
        // below; start those rows on their way to L2 now, so the setup hides
        // part of the first read's latency.
        if (t < kTcRows) {
            const int pti = t / G, ptok = u0.t0 + pti;
            if (pti < kTcRows / G && ptok < u0.qlen) {
                const char* row =
                    reinterpret_cast<const char*>(prm.q + ((size_t)(u0.q0 + ptok) * H + u0.kvh * G + t % G) * D);
#pragma unroll
                for (int x = 0; x < D * 2; x += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + x));
            }
        }
    }

    if (t == 0) {
        *sm_abort = 0;
        for (int i = 0; i < kTcBars; ++i) {
            const bool by_rows = i == kTcBarPReady || i == kTcBarPReady + 1 || i == kTcBarQReady;
            const bool by_k_loads = i < kTcBarKEmpty, by_v_loads = i >= kTcBarVFull && i < kTcBarVEmpty;
            const bool by_all = i == kTcBarUnitEmpty || i == kTcBarUnitEmpty + 1;
            mbar_init(bar(i), by_all ? kTcThreads / 32
                              : by_rows ? kTcSoftmaxWarps
                              : by_k_loads ? kTcKLoadWarps
                              : by_v_loads ? kTcVLoadWarps
                                           : 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tslot)),
                     "r"(S::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    PA_TC_PHASE(1);
    const uint32_t tmem = *tslot;
    const uint32_t tO = tmem;                    // D columns
    const uint32_t tQ = tO + D;                  // D / 2 columns (fp16 pairs)
    const uint32_t tS = tQ + D / 2;              // two score buffers of 64 columns; P(j) over S(j)

    // Units reach the roles through two shared-memory slots.  The first K
    // load warp (the claimer) produces unit u, decoded, into slot u % 2 once
    // every warp has read unit u - 2 from it: the persistent form claims
    // units from the counter, passing over those with nothing to compute
    // (tiles past a sequence's new tokens); the grid form has its own unit,
    // then none.  It produces the next unit kTcClaimAhead key tiles before
    // the end of the current one, so the claim's round trips overlap the
    // tail of the current unit and the claimed tile's Q rows are on their
    // way to L2 before the rows need them.  Every warp consumes the units in
    // order (next_unit).  The grid form takes its unit through a slot too:
    // decoded inside the roles from values the compiler can trace to the
    // block index, the roles' tile loops measured about 20 % slower.
    const bool claimer = warp == kTcLoadWarp0;
    auto produce = [&](int u) {  // claimer warp, all lanes
        const int s = u & 1;
        int id = -1;
        if (lane == 0) {
            TcUnit d = u0;
            if (u < 2 || tc_wait(bar(kTcBarUnitEmpty + s), ((u - 2) >> 1) & 1, limit, sm_abort)) {
                if (!persist) {
                    id = u == 0 ? c0 : -1;
                } else {
                    for (;;) {
                        const unsigned w = atomicAdd(prm.sched, 1u);
                        if (w >= (unsigned)prm.total_units) break;
                        d = tc_unit(prm, (int)w, true);
                        if (d.run) {
                            id = (int)w;
                            break;
                        }
                    }
                }
            } else {
                *sm_abort = 1;
                atomicOr(prm.status, PA_DEV_TIMEOUT);
            }
            sm_unit[s] = id;
            if (id >= 0) sm_units[s] = d;
            mbar_arrive(bar(kTcBarUnitFull + s));
        }
        __syncwarp();  // lane 0's slot writes are visible to the warp
        id = __shfl_sync(kFull, id, 0);
        if (persist && u > 0 && id >= 0) {
            // the claimed tile's Q rows (per token, the G heads' rows are
            // contiguous) on their way to L2
            const TcUnit& d = sm_units[s];
            const int ntok = min(kTcRows / G, d.qlen - d.t0), lines = G * D * 2 / 128;
            const char* q0p = reinterpret_cast<const char*>(prm.q + ((size_t)(d.q0 + d.t0) * H + d.kvh * G) * D);
            for (int i = lane; i < ntok * lines; i += 32)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(q0p + (size_t)(i / lines) * H * D * 2 + (i % lines) * 128));
        }
    };
    // The next unit for the calling warp (all lanes): its number and, in
    // `un`, its decoded fields; -1 when there is none left, -2 when a wait
    // gave up.  `u` counts the units the warp has taken.
    auto next_unit = [&](int& u, TcUnit& un) -> int {
        const int s = u & 1;
        const bool ok = tc_warp_wait(bar(kTcBarUnitFull + s), (u >> 1) & 1, limit, sm_abort);
        const int id = ok ? sm_unit[s] : -2;
        if (id >= 0) un = sm_units[s];
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(bar(kTcBarUnitEmpty + s));
        ++u;
        return id;
    };

    if (warp >= kTcLoadWarp0 && warp < kTcSWarp) {
        // ---------------- load warps: K and V in two independent groups ----------------
        // A TMA instruction occupies its issuing thread for a fixed time
        // whatever the box size, so the copies are spread over many warps:
        // K warp (i, h) copies half h of the 64-column chunks of block i of
        // every K tile, V warp i the blocks i, i + 2 of every V tile (one box
        // each).  Each group
        // walks its own ring and agrees on every wait (one named barrier per
        // group), so a tile is copied by all of a group or by none.
        const int lw = warp - kTcLoadWarp0;
        const bool is_k = lw < kTcKLoadWarps;
        const int i = is_k ? (lw & 3) : lw - kTcKLoadWarps;  // (first) block of the tile
        const int h = is_k ? (lw >> 2) : 0;
        constexpr int kVBlocks = (kTcKeys / kBlockSize) / kTcVLoadWarps;  // V blocks per warp and tile
        constexpr int kHalfChunks = (S::kChunks + 1) / 2;
        const int ch0 = h * kHalfChunks, ch1 = min(S::kChunks, ch0 + kHalfChunks);
        const int slots = is_k ? S::kKSlots : S::kVSlots;
        const int full0 = is_k ? kTcBarKFull : kTcBarVFull, empty0 = is_k ? kTcBarKEmpty : kTcBarVEmpty;
        const int group_bar = is_k ? 1 : 2, group_threads = (is_k ? kTcKLoadWarps : kTcVLoadWarps) * 32;
        bool ok = true;
        int issued = 0;  // tiles issued over all units: ring slot and phase
        int u = 0;
        if (claimer) produce(0);
        for (;;) {
            TcUnit un;
            const int c = next_unit(u, un);
            // the group leaves together, also when one warp's wait gave up
            if (!(ok = tc_group_agree(c != -2, group_bar, group_threads)) || c < 0) break;
            const int nctx = un.nctx, kvh = un.kvh, jb = un.jb;
            const int32_t* bt = prm.block_tables + (size_t)un.b * prm.max_blocks_per_seq;
            auto fetch = [&](int g) {
                const int blk = 32 * g + lane;
                return blk < nctx ? __ldg(bt + blk) : -1;
            };
            // physical block of block blk of the sequence (meaningful for blk < nctx); warp-collective
            TcBlockCursor cur;
            auto lookup = [&](int blk) {
                const int g = blk >> 5;
                if (g != cur.group) {
                    cur.cur = g == cur.group + 1 ? cur.nxt : fetch(g);
                    cur.nxt = fetch(g + 1);
                    cur.group = g;
                }
                return __shfl_sync(kFull, cur.cur, blk & 31);
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
            auto chunk_token = [&](int blk, int p) {
                return p == -2 ? prm.num_tokens : un.q0 + (blk - nctx) * kBlockSize;
            };
            // key tile jt = jb + j of the unit into ring slot x % slots (x
            // counts the tiles of every unit)
            auto issue = [&](int j, int x) {
                const int jt = jb + j;
                if (!is_k) {
                    // blocks i, i + kTcVLoadWarps, ... of the tile, each in one box
                    // laid out [chunk][16 rows][128 B]
                    int phys[kVBlocks];
#pragma unroll
                    for (int y = 0; y < kVBlocks; ++y) phys[y] = lookup(4 * jt + i + y * kTcVLoadWarps);
                    if (lane == 0) {
                        const uint32_t full = bar(full0 + x % slots);
                        mbar_arrive_expect_tx(full, kVBlocks * S::kBlockBytes);
#pragma unroll
                        for (int y = 0; y < kVBlocks; ++y) {
                            const int bi = i + y * kTcVLoadWarps, blk = 4 * jt + bi;
                            const int p = checked(blk, phys[y]);
                            const uint32_t dst =
                                smem_addr(vs + (x % S::kVSlots) * S::kTileBytes) + bi * S::kBlockBytes;
                            if (p >= 0)
                                tma_load_3d(dst, &tmap_vc, 0, (p * prm.num_kv_heads + kvh) * kBlockSize, 0, full);
                            else
                                tc_tma_load_4d(dst, &tmap_vn, 0, kvh, chunk_token(blk, p), 0, full);
                        }
                    }
                    __syncwarp();
                    return;
                }
                const int blk = 4 * jt + i;
                const int phys = lookup(blk);
                if (lane == 0) {
                    const uint32_t full = bar(full0 + x % slots);
                    const int p = checked(blk, phys);
                    // 16-row x 64-column boxes into rows 16 i.. of the slot's
                    // column chunks (the S MMA's operand layout)
                    const uint32_t dst = smem_addr(ks + (x % S::kKSlots) * S::kTileBytes) + i * (kBlockSize * 128);
                    if (ch1 > ch0)
                        mbar_arrive_expect_tx(full, (ch1 - ch0) * (kBlockSize * 128));
                    else
                        mbar_arrive(full);
                    for (int ch = ch0; ch < ch1; ++ch) {
                        if (p >= 0)
                            tma_load_2d(dst + ch * S::kChunkStride, &tmap_kc, ch * 64,
                                        (p * prm.num_kv_heads + kvh) * kBlockSize, full);
                        else
                            tma_load_3d(dst + ch * S::kChunkStride, &tmap_kn, ch * 64, kvh, chunk_token(blk, p), full);
                    }
                }
                __syncwarp();
            };
            cur.group = ((4 * jb) >> 5) - 1;  // the first lookup takes the group read ahead here
            cur.nxt = fetch(cur.group + 1);
            const int jclaim = max(0, un.n - kTcClaimAhead);  // where the claimer produces unit u
            for (int j = 0; j < un.n; ++j) {
                if (claimer && j == jclaim) produce(u);
                // slot `issued` % slots last held the tile issued `slots` tiles
                // earlier: free once the MMA that read it has completed
                const int x = issued;
                if (x >= slots &&
                    !(ok = tc_group_agree(tc_warp_wait(bar(empty0 + x % slots), (x / slots - 1) & 1, limit, sm_abort),
                                          group_bar, group_threads)))
                    break;
                if (lane == 0 && lw == 0) PA_TC_MARK(x, 9);
                if (lane == 0 && lw == kTcKLoadWarps) PA_TC_MARK(x, 11);
                issue(j, x);
                issued = x + 1;
                if (lane == 0 && lw == 0) PA_TC_MARK(x, 10);
                if (lane == 0 && lw == kTcKLoadWarps) PA_TC_MARK(x, 4);
            }
            if (!ok) break;
            if (claimer && un.n == 0) produce(u);  // a part without key tiles
        }
        if (lane == 0) {
            if (!ok && (lw == 0 || lw == kTcKLoadWarps)) {
                *sm_abort = 1;
                atomicOr(prm.status, PA_DEV_TIMEOUT);
            }
            // every copy issued lands before the CTA exits: the whole group
            // issued the same tiles, and a slot holds at most one copy that
            // nobody may have waited for (the latest one)
            for (int x = max(0, issued - slots); x < issued; ++x)
                mbar_wait(bar(full0 + x % slots), (x / slots) & 1, kDefaultWaitLimit);
        }
        __syncwarp();
    } else if (warp == kTcSWarp || warp == kTcPVWarp) {
        // ---------------- MMA warps: lane 0 issues, every lane waits ----------------
        // S and P.V come from two threads so that while one waits for its
        // next inputs the other's MMAs keep the tensor cores busy (each
        // thread's own MMAs run in issue order; the two streams only meet
        // through the barriers below).  x = g + j counts the key tiles of
        // every unit: it picks the ring slots, score buffers and phases.
        bool ok = true;
        int u = 0, g = 0;
        if (warp == kTcSWarp) {
            constexpr uint32_t idS = tc_idesc(kTcRows, kTcKeys, 0);
            const uint64_t kdesc0 = tc_desc(smem_addr(ks), 16, 1024);
            for (int uq = 0;;) {
                TcUnit un;
                const int c = next_unit(u, un);
                if (c < 0) {
                    ok = c != -2;
                    break;
                }
                // the unit's Q rows are in TMEM
                if (!(ok = tc_warp_wait(bar(kTcBarQReady), uq & 1, limit, sm_abort))) break;
                for (int j = 0; j < un.n; ++j) {
                    const int x = g + j;
                    if (lane == 0) PA_TC_MARK(x, 0);
                    // K(x) landed; score buffer x % 2 is free once P.V(x-2), the
                    // last reader of the P written there, has completed
                    if (!(ok = tc_warp_wait(bar(kTcBarKFull + x % S::kKSlots), (x / S::kKSlots) & 1, limit,
                                            sm_abort)))
                        break;
                    if (lane == 0) PA_TC_MARK(x, 14);
                    if (x >= 2 &&
                        !(ok = tc_warp_wait(bar(kTcBarPVDone + (x & 1)), ((x - 2) >> 1) & 1, limit, sm_abort)))
                        break;
                    if (lane == 0) PA_TC_MARK(x, 15);
                    tc_fence_after();
                    if (lane == 0) {
                        // S(x) = Q K(x)^T into score buffer x % 2, Q (A) from TMEM 8
                        // columns per 16 head_dim elements; a descriptor's low field is
                        // the start address / 16, so stepping through a buffer adds
                        // offset / 16
                        const uint64_t kd = kdesc0 + (uint64_t)((x % S::kKSlots) * (S::kTileBytes >> 4));
                        const uint32_t sb = tS + (uint32_t)(x & 1) * kTcKeys;
#pragma unroll
                        for (int k = 0; k < D / 16; ++k)
                            tc_mma_ts(sb, tQ + k * 8,
                                      kd + (uint64_t)(((k >> 2) * S::kChunkStride + (k & 3) * 32) >> 4), idS, k > 0);
                        tc_commit(bar(kTcBarSDone + (x & 1)));
                        tc_commit(bar(kTcBarKEmpty + x % S::kKSlots));
                        PA_TC_MARK(x, 1);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                // Q may be rewritten once the unit's S MMAs have completed
                if (lane == 0) tc_commit(bar(kTcBarQFree));
                __syncwarp();
                g += un.n;
                ++uq;
            }
        } else {
            constexpr uint32_t idO = tc_idesc(kTcRows, D, 1);
            const uint64_t vdesc0 = tc_desc(smem_addr(vs), kBlockSize * 128, 1024);
            for (;;) {
                TcUnit un;
                const int c = next_unit(u, un);
                if (c < 0) {
                    ok = c != -2;
                    break;
                }
                const int partial_tile = un.C % kBlockSize != 0 ? (un.nctx - 1) / 4 : -1;
                for (int j = 0; j < un.n; ++j) {
                    const int x = g + j;
                    if (lane == 0) PA_TC_MARK(x, 12);
                    // rows have written P(x) (and rescaled O if they had to); V(x) landed
                    if (!(ok = tc_warp_wait(bar(kTcBarPReady + (x & 1)), (x >> 1) & 1, limit, sm_abort))) break;
                    if (lane == 0) PA_TC_MARK(x, 2);
                    if (!(ok = tc_warp_wait(bar(kTcBarVFull + x % S::kVSlots), (x / S::kVSlots) & 1, limit,
                                            sm_abort)))
                        break;
                    if (lane == 0) PA_TC_MARK(x, 3);
                    uint8_t* vt = vs + (x % S::kVSlots) * S::kTileBytes;
                    if (un.jb + j == partial_tile) {
                        // V rows of cache slots past the context may hold anything: p is
                        // 0 there, but 0 * NaN is not; clear them before P.V reads them
                        const int bi = (un.nctx - 1) % 4, first = un.C % kBlockSize;
                        const int units = (kBlockSize - first) * S::kChunks * 8;
                        uint8_t* vb = vt + bi * S::kBlockBytes;
                        for (int y = lane; y < units; y += 32) {
                            const int r = first + y / (S::kChunks * 8), w = y % (S::kChunks * 8);
                            *reinterpret_cast<uint4*>(vb + (w >> 3) * (kBlockSize * 128) + r * 128 + (w & 7) * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        // O += P(x) V(x), P over S(x) in score buffer x % 2, one MMA
                        // per block of 16 keys (V block: 64-column chunks 2 KB apart,
                        // 8-key groups 1 KB apart); score buffer x % 2 and V slot
                        // x % kVSlots are free when they complete.  The unit's first
                        // tile overwrites O.
                        const uint64_t vd = vdesc0 + (uint64_t)((x % S::kVSlots) * (S::kTileBytes >> 4));
                        const uint32_t a = tS + (uint32_t)(x & 1) * kTcKeys;
#pragma unroll
                        for (int k = 0; k < kTcKeys / 16; ++k)
                            tc_mma_ts(tO, a + k * 8, vd + (uint64_t)((k * S::kBlockBytes) >> 4), idO, (j > 0 || k > 0));
                        tc_commit(bar(kTcBarPVDone + (x & 1)));
                        tc_commit(bar(kTcBarVEmpty + x % S::kVSlots));
                        PA_TC_MARK(x, 13);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                g += un.n;
            }
        }
        if (lane == 0) {
            if (!ok) {
                *sm_abort = 1;
                atomicOr(prm.status, PA_DEV_TIMEOUT);
            }
            // every MMA this thread issued has completed once this commit arrives
            const uint32_t drain = bar(warp == kTcSWarp ? kTcBarSDrain : kTcBarPVDrain);
            tc_commit(drain);
            mbar_wait(drain, 0, kDefaultWaitLimit);
        }
        __syncwarp();
    } else {
        // ---------------- softmax warps: thread t owns row t (TMEM lane t) ----------------
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const int ti = t / G;
        const float sl2 = prm.scale_log2;
        // Q row (token ti of the unit's tile, head kvh * G + t % G) into TMEM
        // columns tQ.., two halves per column; rows that do not exist hold zeros
        auto load_q = [&](const TcUnit& un) {
            const int my_tok = un.t0 + ti;
            const bool row_real = ti < kTcRows / G && my_tok < un.qlen;
            // two 32-column chunks (16 loads) in flight per round: the row
            // arrives in D / 128 round trips instead of D / 64
            const uint4* qrow =
                reinterpret_cast<const uint4*>(prm.q + ((size_t)(un.q0 + my_tok) * H + un.kvh * G + t % G) * D);
            constexpr int kPer = D / 2 >= 64 ? 2 : 1;  // chunks per round
#pragma unroll 1
            for (int c0 = 0; c0 < D / 2; c0 += 32 * kPer) {
                uint32_t v[kPer][32];
#pragma unroll
                for (int h = 0; h < kPer; ++h)
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint4 x = row_real ? __ldg(qrow + (c0 + 32 * h) / 4 + u) : make_uint4(0u, 0u, 0u, 0u);
                        v[h][4 * u] = x.x;
                        v[h][4 * u + 1] = x.y;
                        v[h][4 * u + 2] = x.z;
                        v[h][4 * u + 3] = x.w;
                    }
                if constexpr (kPer == 2)
                    tc_st32x2(tQ + lane_off + c0, v[0], tQ + lane_off + c0 + 32, v[1]);
                else
                    tc_st32(tQ + lane_off + c0, v[0]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kTcBarQReady));
        };
        // the next unit, or -1 / -2 (see next_unit)
        int u = 0;
        auto next_run = [&](TcUnit& un) -> int { return next_unit(u, un); };
        TcUnit cur;
        int rc = next_run(cur);
        bool ok = rc != -2;
        if (rc >= 0) load_q(cur);
        PA_TC_PHASE(2);
        for (int g = 0, uq = 0; ok && rc >= 0; ++uq) {
            // the fields the epilogue needs wait in shared memory, not in
            // registers, while the tile loop runs
            if (lane == 0) rows_units[warp] = cur;
            __syncwarp();
            const int my_tok = cur.t0 + ti;  // chunk token index of the row
            const int n = cur.n, jb = cur.jb, nctx = cur.nctx, C = cur.C;
            float m = -INFINITY, l = 0.f;  // reference max (scaled, log2 domain) and exp sum
            for (int j = 0; j < n; ++j) {
                const int x = g + j;
                const uint32_t sb = tS + (uint32_t)(x & 1) * kTcKeys + lane_off;  // this row of score buffer x % 2
                if (!(ok = tc_warp_wait(bar(kTcBarSDone + (x & 1)), (x >> 1) & 1, limit, sm_abort))) break;
                tc_fence_after();
                if (t == 0) PA_TC_MARK(x, 5);
                uint32_t sv[2][32];
                tc_ld32x2(sb, sv[0], sb + 32, sv[1]);
                // visibility: every key of a tile made only of full context blocks
                // is visible; otherwise mask per key
                const int jt = jb + j;
                const bool full_ctx = 4 * jt + 3 < nctx - (C % kBlockSize != 0 ? 1 : 0);
                if (!full_ctx) {
                    // visible slots of each 16-key block of the tile for this row:
                    // a context block shows its keys below C, a chunk block the
                    // chunk tokens up to the row's own; then one compare per key
                    // against its (compile-time) slot
                    int nvis[4];
#pragma unroll
                    for (int qb = 0; qb < 4; ++qb) {
                        const int blk = 4 * jt + qb;
                        const int vis = blk < nctx ? C - blk * kBlockSize : my_tok + 1 - (blk - nctx) * kBlockSize;
                        nvis[qb] = min(max(vis, 0), kBlockSize);
                    }
                    const uint32_t hidden = __float_as_uint(sl2 >= 0.f ? -INFINITY : INFINITY);
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (((h2 * 32 + c) & 15) >= nvis[(h2 * 32 + c) >> 4]) sv[h2][c] = hidden;
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
                // P(x) over S(x), which is in registers now: the S MMA of this
                // buffer was issued after P.V(x-2), the buffer's previous reader,
                // had completed, and the next one waits for P.V(x)
                tc_st32(sb, pk);
                if (j > 0 && __any_sync(kFull, move)) {
                    // O is written by P.V(x-1): wait for it, then rescale this row
                    // (P.V(x-3) was waited for one tile ago).  The unit's first
                    // tile needs none: its P.V overwrites O.
                    if (!(ok = tc_warp_wait(bar(kTcBarPVDone + ((x - 1) & 1)), ((x - 1) >> 1) & 1, limit, sm_abort)))
                        break;
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
                if (t == 0) PA_TC_MARK(x, 6);
                if (t == 96) PA_TC_MARK(x, 7);
                if (lane == 0) mbar_arrive(bar(kTcBarPReady + (x & 1)));
            }
            PA_TC_PHASE(3);
            if (!ok) break;
            // Where this row's result goes (the unit's fields are dead after
            // the next unit is taken): the fp16 output row, or the part's
            // partial slot of a key split
            const TcUnit cu = rows_units[warp];
            const bool row_real = ti < kTcRows / G && cu.t0 + ti < cu.qlen;
            const int part = cu.part;
            const size_t slot = part >= 0 ? ((size_t)cu.unit_r * prm.split_parts + part) * kTcRows + t : 0;
            __half* orow_h = prm.out + ((size_t)(cu.q0 + cu.t0 + ti) * H + cu.kvh * G + (t % G)) * D;
            // The next unit's Q goes into TMEM while this unit's last P.Vs run:
            // its S MMAs then start while the rows store this unit's O.
            TcUnit nxt;
            PA_TC_PHASE(8);
            const int rn = next_run(nxt);
            if (rn == -2) {
                ok = false;
                break;
            }
            if (rn >= 0) {
                PA_TC_PHASE(9);
                if (!(ok = tc_warp_wait(bar(kTcBarQFree), uq & 1, limit, sm_abort))) break;
                tc_fence_after();
                PA_TC_PHASE(10);
                load_q(nxt);
                PA_TC_PHASE(11);
            }
            // the last two P.Vs of the unit (one per score buffer) complete before O is read
            const int xe = g + n;
            if (n >= 2) ok = tc_warp_wait(bar(kTcBarPVDone + ((xe - 2) & 1)), ((xe - 2) >> 1) & 1, limit, sm_abort);
            if (ok && n >= 1) ok = tc_warp_wait(bar(kTcBarPVDone + ((xe - 1) & 1)), ((xe - 1) >> 1) & 1, limit, sm_abort);
            if (!ok) break;
            if (rn >= 0) PA_TC_PHASE(12);
            tc_fence_after();
            if (part >= 0) {
                // a part of a key split: the row's partial (m, l and O relative to
                // 2^m, fp32) for the merge; a part without key tiles leaves m = -inf
                // and l = 0, which the merge skips without reading its O
                if (row_real) {
                    prm.split_ml[2 * slot] = m;
                    prm.split_ml[2 * slot + 1] = l;
                }
                float4* orow = reinterpret_cast<float4*>(prm.split_o + slot * D);
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 64) {
                    uint32_t ov[2][32];
                    tc_ld32x2(tO + lane_off + c0, ov[0], tO + lane_off + c0 + 32, ov[1]);
                    if (row_real && n > 0) {
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int c = 0; c < 32; c += 4)
                                orow[(c0 + 32 * h + c) / 4] =
                                    make_float4(__uint_as_float(ov[h][c]), __uint_as_float(ov[h][c + 1]),
                                                __uint_as_float(ov[h][c + 2]), __uint_as_float(ov[h][c + 3]));
                    }
                }
            } else {
                // O / l to fp16 for the rows that exist
                const float inv = 1.f / l;
                // two 32-column chunks per wait::ld
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 64) {
                    uint32_t ov[2][32];
                    tc_ld32x2(tO + lane_off + c0, ov[0], tO + lane_off + c0 + 32, ov[1]);
                    if (row_real) {
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int c = 0; c < 32; c += 8) {
                                uint4 w;
                                uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    wp[e] = half2_bits(__floats2half2_rn(__uint_as_float(ov[h][c + 2 * e]) * inv,
                                                                         __uint_as_float(ov[h][c + 2 * e + 1]) * inv));
                                *reinterpret_cast<uint4*>(orow_h + c0 + 32 * h + c) = w;
                            }
                    }
                }
            }
            // O has been read (tcgen05.ld waited): the next unit's first P.V,
            // which waits for these rows' P, may overwrite it
            tc_fence_before();
            if (rn >= 0) PA_TC_PHASE(13);
            g += n;
            cur = nxt;
            rc = rn;
        }
        if (!ok && lane == 0) {
            *sm_abort = 1;
            atomicOr(prm.status, PA_DEV_TIMEOUT);
        }
    }
    PA_TC_PHASE(4);
    tc_fence_before();
    __syncthreads();  // every role done: no copy or MMA in flight past this point
    PA_TC_PHASE(5);
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(S::kTmemCols));
    if (persist && t == 0) {
        // The last CTA to finish re-arms the counter for the next call: every
        // claim of every CTA precedes its ticket.
        __threadfence();
        if (atomicAdd(prm.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(prm.sched, 0u);
            atomicExch(prm.sched + 1, 0u);
            __threadfence();
        }
    }
}

// Merge of a key split (PrefixParams::split_parts): every row of split unit
// r had its keys walked in split_parts ranges, each leaving (m_p, l_p, O_p)
// with O_p and l_p relative to 2^m_p (m in the scaled log2 domain).  The
// output is the log-sum-exp merge of the decode path's reduce, here over the
// key ranges of one query tile: with M = max_p m_p and w_p = 2^(m_p - M),
//     out = sum_p w_p O_p / sum_p w_p l_p,
// folded in part order.  A part with m_p = -inf saw no key of the row and
// weighs nothing (its O is not read).  Grid (split units, row groups); a
// thread takes 4 columns of one row.
template <int D>
__global__ void __launch_bounds__(256) pa_prefix_merge_kernel(const PrefixParams prm) {
    constexpr int kCols = D / 4;               // float4 columns of a row
    constexpr int kRowsPerCta = 256 / kCols;   // 4 at head_dim 256
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int r = blockIdx.x, w = prm.split_whole + r;
    const int tile = w % prm.tiles_per_seq, kvh = (w / prm.tiles_per_seq) % prm.num_kv_heads;
    const int b = w / (prm.tiles_per_seq * prm.num_kv_heads);
    const int G = prm.group, H = prm.num_heads, tile_tokens = kTcRows / G;
    // the same checks as the kernel that wrote the partials: a unit it left
    // is left here too
    const int C = __ldg(prm.context_lens + b);
    const int q0 = __ldg(prm.query_start_loc + b), q1 = __ldg(prm.query_start_loc + b + 1);
    const int qlen = q1 - q0;
    if (C < 0 || C > prm.max_context_len || C > prm.max_blocks_per_seq * kBlockSize || qlen < 0 ||
        qlen > prm.max_query_len || q0 < 0 || q1 > prm.num_tokens)
        return;
    const int row = blockIdx.y * kRowsPerCta + (int)threadIdx.x / kCols, col = (int)threadIdx.x % kCols;
    const int ti = row / G, tok = tile * tile_tokens + ti;
    if (ti >= tile_tokens || tok >= qlen) return;
    const int k = prm.split_parts;
    const size_t slot0 = (size_t)r * k * kTcRows + row;  // part p: slot0 + p * kTcRows
    float M = -INFINITY;
    for (int p = 0; p < k; ++p) M = fmaxf(M, prm.split_ml[2 * (slot0 + (size_t)p * kTcRows)]);
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = 0; p < k; ++p) {
        const size_t slot = slot0 + (size_t)p * kTcRows;
        const float mp = prm.split_ml[2 * slot];
        if (mp == -INFINITY) continue;
        const float wp = exp2f(mp - M);
        den += wp * prm.split_ml[2 * slot + 1];
        const float4 o = reinterpret_cast<const float4*>(prm.split_o + slot * D)[col];
        acc.x += wp * o.x;
        acc.y += wp * o.y;
        acc.z += wp * o.z;
        acc.w += wp * o.w;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __half2* dst = reinterpret_cast<__half2*>(prm.out + ((size_t)(q0 + tok) * H + kvh * G + row % G) * D + 4 * col);
    dst[0] = __floats2half2_rn(acc.x * inv, acc.y * inv);
    dst[1] = __floats2half2_rn(acc.z * inv, acc.w * inv);
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
constexpr int tc_ctas_per_sm() {
    constexpr int by_smem = (228 * 1024) / (PrefixTcShape<D>::kSmemBytes + 1024);
    constexpr int by_tmem = 512 / PrefixTcShape<D>::kTmemCols;
    constexpr int by_threads = 2048 / kTcThreads;
    constexpr int by_regs = 65536 / (kTcThreads * kTcMaxRegs);  // the kernel may use all kTcMaxRegs
    constexpr int a = by_smem < by_tmem ? by_smem : by_tmem, b = by_threads < by_regs ? by_threads : by_regs;
    return a < b ? a : b;
}
}  // namespace

int prefix_tc_ctas_per_sm(int head_dim) {
    switch (head_dim) {
        case 64: return tc_ctas_per_sm<64>();
        case 128: return tc_ctas_per_sm<128>();
        case 256: return tc_ctas_per_sm<256>();
        default: return -1;
    }
}

namespace {
template <int D>
cudaError_t launch_prefix_tc_t(const PrefixParams& prm, const CUtensorMap* maps, dim3 grid, cudaStream_t stream) {
    const int smem = PrefixTcShape<D>::kSmemBytes;
    static std::atomic<unsigned long long> done{0};
    cudaError_t e = once_per_device(done, [&] {
        cudaError_t r = cudaFuncSetAttribute(pa_prefix_tc_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(pa_prefix_tc_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        return r;
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = prm.sched ? cudaLaunchKernelEx(&cfg, pa_prefix_tc_kernel<D, true>, maps[0], maps[1], maps[2], maps[3], prm)
                  : cudaLaunchKernelEx(&cfg, pa_prefix_tc_kernel<D, false>, maps[0], maps[1], maps[2], maps[3], prm);
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

namespace {
template <int D>
cudaError_t launch_prefix_merge_t(const PrefixParams& prm, int units, cudaStream_t stream) {
    constexpr int kRowsPerCta = 256 / (D / 4);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units, kTcRows / kRowsPerCta, 1);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, pa_prefix_merge_kernel<D>, prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_prefix_merge(int head_dim, const PrefixParams& prm, int units, cudaStream_t stream) {
    static_assert(kPrefixTileRows == kTcRows, "split workspace rows");
    switch (head_dim) {
        case 64: return launch_prefix_merge_t<64>(prm, units, stream);
        case 128: return launch_prefix_merge_t<128>(prm, units, stream);
        case 256: return launch_prefix_merge_t<256>(prm, units, stream);
        default: return cudaErrorInvalidValue;
    }
}
