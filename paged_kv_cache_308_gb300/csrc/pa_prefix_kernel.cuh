// Chunked-prefill ("prefix") attention over the paged cache, for GB300.
// Included by pa_prefix.cu.
//
// Sequence b has context_lens[b] tokens in the paged cache and brings a chunk
// of q_len_b new tokens (rows query_start_loc[b] .. [b+1]-1 of q, k_new,
// v_new).  New token i attends to all context tokens and to chunk tokens
// 0..i.  This is the prefix path of the "qwen3_6_scripts/paged_attn.py"
// commit page: online softmax over the pre-gathered paged context, then over
// the current chunk with the same update; here both key sources stream
// through one shared-memory ring and one running softmax state per row.
//
// Mapping:
// * one CTA per (query tile, kv head, sequence); 4 warps x 16 rows.  Row r is
//   (token r / G, head r % G) of the tile, so a tile holds floor(64 / G) new
//   tokens and every K/V block is loaded once for all heads of the group;
// * K/V blocks of 16 tokens arrive by 2-D TMA boxes (context, through the
//   block table) or 3-D boxes (chunk, [token][kv head][dim]); all with the
//   128-byte swizzle, in a ring of kPrefixStages stages with "full" (copy
//   landed) and "empty" (all warps done) mbarriers; warp 0 lane 0 issues;
// * S = Q K^T and O += P V run as m16n8k16 MMAs, FlashAttention-2 style: the
//   S accumulator fragments become the A fragments of P after rounding to
//   fp16; Q stays in shared memory (swizzled) and is re-read per k-step;
// * every wait is bounded; a wait that gives up sets PA_DEV_TIMEOUT, the
//   issuing lane drains its copies, and the CTA exits without writing.

constexpr int kPrefixWarps = 4;
constexpr int kPrefixRows = kPrefixWarps * 16;
constexpr int kPrefixStages = 4;

template <int D>
struct PrefixShape {
    static constexpr int kSteps = D / 16;
    static constexpr int kChunks = D / 64;
    static constexpr int kBoxBytes = kBlockSize * 128;
    static constexpr int kTileBytes = kBlockSize * D * 2;
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kQBytes = kPrefixRows * D * 2;
    static constexpr int kStageArea = kPrefixStages * kStageBytes;
    static constexpr int kCtrlBytes = 2 * kPrefixStages * 8 + kPrefixStages * 4 + 16;
    static constexpr int kSmemBytes = 1024 + kStageArea + kQBytes + kCtrlBytes;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget of one CTA");
};

// Byte offset of 16-byte unit u of row r in the Q tile (rows of D halves,
// unit index XOR row mod 8 so that ldmatrix rows hit distinct bank groups).
template <int D>
__device__ __forceinline__ uint32_t q_swz(int r, int u) {
    return static_cast<uint32_t>(r * (D * 2) + ((u ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kPrefixWarps * 32, 1)
    pa_prefix_kernel(const __grid_constant__ CUtensorMap tmap_kc, const __grid_constant__ CUtensorMap tmap_vc,
                     const __grid_constant__ CUtensorMap tmap_kn, const __grid_constant__ CUtensorMap tmap_vn,
                     const PrefixParams prm) {
    using S = PrefixShape<D>;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* qtile = smem + S::kStageArea;
    uint64_t* full = reinterpret_cast<uint64_t*>(qtile + S::kQBytes);
    uint64_t* empty = full + kPrefixStages;
    int* stage_ok = reinterpret_cast<int*>(empty + kPrefixStages);
    int* sm_abort = stage_ok + kPrefixStages;

    const int tile = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = prm.group, H = prm.num_heads;
    const int tile_tokens = kPrefixRows / G;

    const int C = __ldg(prm.context_lens + b);
    const int q0 = __ldg(prm.query_start_loc + b), q1 = __ldg(prm.query_start_loc + b + 1);
    const int qlen = q1 - q0;
    if (C < 0 || C > prm.max_context_len || C > prm.max_blocks_per_seq * kBlockSize || qlen < 0 ||
        qlen > prm.max_query_len || q0 < 0 || q1 > prm.num_tokens) {
        if (tile == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(prm.status, PA_DEV_BAD_SEQ_LEN);
        return;
    }
    const int t0 = tile * tile_tokens;  // first chunk token of this tile
    if (t0 >= qlen) return;
    const int tlast = min(qlen, t0 + tile_tokens) - 1;
    const int nctx = (C + kBlockSize - 1) / kBlockSize;
    const int nblocks = nctx + tlast / kBlockSize + 1;  // context blocks, then chunk blocks up to tlast
    const int32_t* bt = prm.block_tables + (size_t)b * prm.max_blocks_per_seq;

    const uint32_t stage0 = smem_addr(smem);
    const uint32_t full0 = smem_addr(full), empty0 = smem_addr(empty);
    if (threadIdx.x == 0) {
        *sm_abort = 0;
        for (int s = 0; s < kPrefixStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kPrefixWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }

    // Producer: stage block `it` (context blocks first, then chunk blocks).
    auto issue = [&](int it) {
        const int s = it % kPrefixStages;
        const uint32_t bar = full0 + 8 * s;
        const uint32_t kdst = stage0 + s * S::kStageBytes, vdst = kdst + S::kTileBytes;
        if (it < nctx) {
            const int phys = __ldg(bt + it);
            const bool ok = phys >= 0 && (long long)phys < prm.num_blocks;
            stage_ok[s] = ok;
            if (ok) {
                mbar_arrive_expect_tx(bar, S::kStageBytes);
                const int row = (phys * prm.num_kv_heads + kvh) * kBlockSize;
#pragma unroll
                for (int ch = 0; ch < S::kChunks; ++ch) {
                    tma_load_2d(kdst + ch * S::kBoxBytes, &tmap_kc, ch * 64, row, bar);
                    tma_load_2d(vdst + ch * S::kBoxBytes, &tmap_vc, ch * 64, row, bar);
                }
            } else {
                atomicOr(prm.status, PA_DEV_BAD_BLOCK_ID);
                mbar_arrive(bar);
            }
        } else {
            stage_ok[s] = 1;
            mbar_arrive_expect_tx(bar, S::kStageBytes);
            const int tok = q0 + (it - nctx) * kBlockSize;
#pragma unroll
            for (int ch = 0; ch < S::kChunks; ++ch) {
                tma_load_3d(kdst + ch * S::kBoxBytes, &tmap_kn, ch * 64, kvh, tok, bar);
                tma_load_3d(vdst + ch * S::kBoxBytes, &tmap_vn, ch * 64, kvh, tok, bar);
            }
        }
    };

    const bool producer = threadIdx.x == 0;
    int issued = 0;  // blocks issued so far (meaningful in the producer lane)
    if (producer)
        for (; issued < kPrefixStages && issued < nblocks; ++issued) issue(issued);

    // Q tile: row r = (token t0 + r / G, head kvh * G + r % G); rows past the
    // chunk or past the group are zero.
    for (int idx = threadIdx.x; idx < kPrefixRows * (D / 8); idx += blockDim.x) {
        const int r = idx / (D / 8), u = idx % (D / 8);
        const int ti = r / G, h = r % G;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (ti < tile_tokens && t0 + ti < qlen)
            v = __ldg(reinterpret_cast<const uint4*>(prm.q + ((size_t)(q0 + t0 + ti) * H + kvh * G + h) * D) + u);
        *reinterpret_cast<uint4*>(qtile + q_swz<D>(r, u)) = v;
    }
    __syncthreads();


    const int g = lane >> 2, c = lane & 3;
    const int row0 = warp * 16 + g, row1 = row0 + 8;                  // rows of this lane
    const int tok_r0 = t0 + row0 / G, tok_r1 = t0 + row1 / G;         // their chunk token index
    const float sl2 = prm.scale_log2;
    const int mi = lane >> 3, r8 = lane & 7;
    // ldmatrix lane roles: A (Q rows), B (K rows = keys), B^T (V rows = keys)
    const int qa_row = warp * 16 + r8 + ((mi & 1) << 3), qa_u = mi >> 1;
    const int kb_key = r8 + ((mi >> 1) << 3), kb_u = mi & 1;
    const int vb_key = r8 + ((mi & 1) << 3), vb_u = mi >> 1;

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows row0, row1

    // A wait that gives up puts the warp in abort mode: it skips the rest of
    // its waits and math but keeps the loop (and the block-wide barriers of
    // partial context blocks) in step with the other warps.
    bool aborted = false;
    for (int it = 0; it < nblocks; ++it) {
        const int s = it % kPrefixStages;
        if (!aborted) {
            const bool ok = !prm.force_timeout && mbar_wait(full0 + 8 * s, (it / kPrefixStages) & 1, prm.wait_limit);
            aborted = !__all_sync(kFull, ok);
            if (aborted && lane == 0) atomicExch(sm_abort, 1);
        }
        const bool ctx = it < nctx;
        const uint32_t kst = stage0 + s * S::kStageBytes, vst = kst + S::kTileBytes;
        const int nvalid_ctx = ctx ? min(kBlockSize, C - it * kBlockSize) : kBlockSize;
        if (ctx && nvalid_ctx < kBlockSize) {
            // cache slots past the context may hold anything: clear those V rows
            // once (all warps wait for it) so that 0 * NaN cannot reach O
            __syncthreads();
            if (!*sm_abort) {
                uint8_t* vgen = smem + (vst - stage0);
                const int units = (kBlockSize - nvalid_ctx) * S::kChunks * 8;
                for (int u = threadIdx.x; u < units; u += blockDim.x) {
                    const int r = nvalid_ctx + u / (S::kChunks * 8), rem = u % (S::kChunks * 8);
                    *reinterpret_cast<uint4*>(vgen + (rem >> 3) * S::kBoxBytes + r * 128 + (rem & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            __syncthreads();
        }
        if (aborted) continue;
        if (stage_ok[s]) {
            // S = Q K^T for this warp's 16 rows and the block's 16 keys
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < S::kSteps; ++ks) {
                uint32_t a[4], kb[4];
                ldsm_x4(a, smem_addr(qtile) + q_swz<D>(qa_row, 2 * ks + qa_u));
                ldsm_x4(kb, kst + (ks >> 2) * S::kBoxBytes + swz(kb_key, ((ks & 3) << 1) + kb_u));
                mma_16816(sa, a, kb[0], kb[1]);  // keys 0..7
                mma_16816(sb, a, kb[2], kb[3]);  // keys 8..15
            }
            // lane holds rows row0 (sa/sb [0], [1]) and row1 ([2], [3]) at keys 2c, 2c+1 (+8)
            float sc[8] = {sa[0], sa[1], sb[0], sb[1], sa[2], sa[3], sb[2], sb[3]};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int key = (e & 2 ? 8 : 0) + 2 * c + (e & 1);
                const int tokr = e < 4 ? tok_r0 : tok_r1;
                const bool ok = ctx ? key < nvalid_ctx : ((it - nctx) * kBlockSize + key <= tokr);
                sc[e] = ok ? sc[e] * sl2 : -INFINITY;
            }
            float mx0 = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
            float mx1 = fmaxf(fmaxf(sc[4], sc[5]), fmaxf(sc[6], sc[7]));
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            // a row with no visible key yet keeps alpha = 1 and p = 0
            const float base0 = mn0 == -INFINITY ? 0.f : mn0, base1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = exp2f(m0 - base0), al1 = exp2f(m1 - base1);
            m0 = mn0;
            m1 = mn1;
            const __half2 p00 = __floats2half2_rn(exp2f(sc[0] - base0), exp2f(sc[1] - base0));  // row0 keys 2c..
            const __half2 p01 = __floats2half2_rn(exp2f(sc[2] - base0), exp2f(sc[3] - base0));  // row0 keys 8+2c..
            const __half2 p10 = __floats2half2_rn(exp2f(sc[4] - base1), exp2f(sc[5] - base1));  // row1 keys 2c..
            const __half2 p11 = __floats2half2_rn(exp2f(sc[6] - base1), exp2f(sc[7] - base1));  // row1 keys 8+2c..
            const float2 f00 = __half22float2(p00), f01 = __half22float2(p01);
            const float2 f10 = __half22float2(p10), f11 = __half22float2(p11);
            l0 = l0 * al0 + (f00.x + f00.y + f01.x + f01.y);
            l1 = l1 * al1 + (f10.x + f10.y + f11.x + f11.y);
            if (__any_sync(kFull, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt) {
                    o[nt][0] *= al0;
                    o[nt][1] *= al0;
                    o[nt][2] *= al1;
                    o[nt][3] *= al1;
                }
            }
            // P as the A operand (16 rows x 16 keys): the accumulator layout of S
            const uint32_t pa[4] = {half2_bits(p00), half2_bits(p10), half2_bits(p01), half2_bits(p11)};
            // O += P V
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                uint32_t vb[4];
                ldsm_x4_trans(vb, vst + (dp >> 2) * S::kBoxBytes + swz(vb_key, ((dp & 3) << 1) + vb_u));
                mma_16816(o[2 * dp], pa, vb[0], vb[1]);
                mma_16816(o[2 * dp + 1], pa, vb[2], vb[3]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        // the producer refills this stage once every warp has released it
        if (warp == 0) {
            int ok = 1;
            if (lane == 0 && issued < nblocks) {
                ok = mbar_wait(empty0 + 8 * (issued % kPrefixStages), ((issued / kPrefixStages) - 1) & 1,
                               prm.wait_limit);
                if (ok) {
                    issue(issued);
                    ++issued;
                }
            }
            aborted = !__shfl_sync(kFull, ok, 0);
            if (aborted && lane == 0) atomicExch(sm_abort, 1);
        }
    }

    if (aborted) {
        if (lane == 0) {
            atomicOr(prm.status, PA_DEV_TIMEOUT);
            atomicExch(sm_abort, 1);
        }
        // drain the copies still in flight: the last one issued on each stage
        if (producer)
            for (int k = issued > kPrefixStages ? issued - kPrefixStages : 0; k < issued; ++k)
                mbar_wait(full0 + 8 * (k % kPrefixStages), (k / kPrefixStages) & 1, kDefaultWaitLimit);
    }
    __syncthreads();
    if (*sm_abort) return;

    // Row sums over the quad, then O / l to fp16 for the rows that exist.
    l0 += __shfl_xor_sync(kFull, l0, 1);
    l0 += __shfl_xor_sync(kFull, l0, 2);
    l1 += __shfl_xor_sync(kFull, l1, 1);
    l1 += __shfl_xor_sync(kFull, l1, 2);
    const float inv0 = 1.f / l0, inv1 = 1.f / l1;
    const bool w0 = row0 / G < tile_tokens && tok_r0 < qlen, w1 = row1 / G < tile_tokens && tok_r1 < qlen;
    __half* out0 = prm.out + ((size_t)(q0 + tok_r0) * H + kvh * G + row0 % G) * D;
    __half* out1 = prm.out + ((size_t)(q0 + tok_r1) * H + kvh * G + row1 % G) * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
        const int d = nt * 8 + 2 * c;
        if (w0) *reinterpret_cast<__half2*>(out0 + d) = __floats2half2_rn(o[nt][0] * inv0, o[nt][1] * inv0);
        if (w1) *reinterpret_cast<__half2*>(out1 + d) = __floats2half2_rn(o[nt][2] * inv1, o[nt][3] * inv1);
    }
}

int prefix_smem_bytes(int head_dim) {
    switch (head_dim) {
        case 64: return PrefixShape<64>::kSmemBytes;
        case 128: return PrefixShape<128>::kSmemBytes;
        case 256: return PrefixShape<256>::kSmemBytes;
        default: return -1;
    }
}

namespace {
template <int D>
cudaError_t launch_prefix_t(const PrefixParams& prm, const CUtensorMap* maps, dim3 grid, cudaStream_t stream) {
    const int smem = PrefixShape<D>::kSmemBytes;
    static std::atomic<unsigned long long> done{0};
    cudaError_t e = once_per_device(done, [&] {
        return cudaFuncSetAttribute(pa_prefix_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kPrefixWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, pa_prefix_kernel<D>, maps[0], maps[1], maps[2], maps[3], prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_prefix(int head_dim, const PrefixParams& prm, const CUtensorMap* maps, dim3 grid,
                          cudaStream_t stream) {
    switch (head_dim) {
        case 64: return launch_prefix_t<64>(prm, maps, grid, stream);
        case 128: return launch_prefix_t<128>(prm, maps, grid, stream);
        case 256: return launch_prefix_t<256>(prm, maps, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}
