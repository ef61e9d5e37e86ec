// C-ABI layer of the paged-attention decode library: argument validation,
// host dispatch (single-pass vs split-KV), the cached workspace, tensor maps
// and kernel launches.  The public contract is include/pa_decode.h.
//
// Dispatch follows the decode dispatch of the "qwen3_6_scripts/paged_attn.py"
// commit page (a single-CTA kernel for short sequences, the partitioned kernel
// plus a reduce for long ones); the thresholds are this library's own, set
// from GB300 measurements rather than the page's 8192-token rule.  The cached
// workspace follows that page's allocate-once, reuse-across-calls advice.
#include "pa_decode.h"

#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "pa_internal.h"
#include "pa_prefix.h"

namespace {

constexpr int kDefaultPartition = 512;
constexpr int kOneWavePoolMinPartition = 2048;  // see make_plan
constexpr int kOneWaveMinLen = 128;              // see make_plan
constexpr int kOneWaveShortMinParts = 4;         // see make_plan
constexpr int kOneWaveShortMaxPartition = 128;  // see make_plan
// SM count assumed by pa_decode_workspace_size when no device answers (above any GPU's)
constexpr int kMaxSmsBound = 1024;
// choose_shape: 2x2 CTAs for batches of at least kManyPairs (sequence, kv
// head) pairs whose longest sequence has at most kManyPairsMaxLen tokens
constexpr long long kManyPairs = 64;
constexpr int kManyPairsMaxLen = 16384;
// PA_MODE_PERSISTENT CTA shapes: 4 x 2 when the scan apportions the partitions
// (about one item per CTA), 1 x 2 for a caller's partition size (many items)
constexpr int kPersistentWarps = 4, kPersistentWarpsFixedSize = 1, kPersistentStages = 2;
constexpr int kMaxDevices = 64;
constexpr size_t kWsAlign = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t split_workspace_bytes(long long num_seqs, long long num_heads, long long max_partitions, long long head_dim) {
    if (max_partitions <= 1) return 0;
    const size_t rows = static_cast<size_t>(num_seqs) * num_heads * max_partitions;
    return align_up(rows * 4, kWsAlign) * 2 + align_up(rows * head_dim * 4, kWsAlign);
}

// Bytes of the pooled split's claim counters, one u64 per (sequence, kv head);
// they sit right after the partials.
size_t claims_bytes(long long num_seqs, long long num_kv_heads) {
    return align_up(static_cast<size_t>(num_seqs) * num_kv_heads * 8, kWsAlign);
}

// The fused combine also keeps two u32 words per (sequence, kv head): the
// ticket (or, merging in parallel, the arrivals) and the departures.  They
// sit after a slot the size of the claim counters, so that a pooled split
// call of the same shape on the same workspace (which arms those counters)
// never touches them.
size_t fused_workspace_bytes(long long num_seqs, long long num_heads, long long num_kv_heads,
                             long long max_partitions, long long head_dim) {
    if (max_partitions <= 1) return 0;
    return split_workspace_bytes(num_seqs, num_heads, max_partitions, head_dim) +
           claims_bytes(num_seqs, num_kv_heads) + align_up(static_cast<size_t>(num_seqs) * num_kv_heads * 8, kWsAlign);
}

// SM count of the current device, cached per device.
int query_sm_count(int* num_sms) {
    static int cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices && cached[dev] > 0) {
        *num_sms = cached[dev];
        return PA_OK;
    }
    if (cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) cached[dev] = *num_sms;
    return PA_OK;
}

// Head_dim slice of one reduce CTA: the widest slice that still gives the
// reduce grid about two CTAs per SM, so a large batch runs few, wide CTAs
// (short launch and latency chains) and a single long sequence runs narrow
// ones (more loads in flight per partial).  Two rather than four CTAs per
// SM: b8_u8192 27.33 -> 27.05 us per call (128-wide slices instead of 64),
// b4_l32768_peaked 85.26 -> 85.41 (64 instead of 32), the rest unchanged.
// 4-warp CTAs per SM in a one-wave plan: enough to keep about 128 KB of
// K/V copies in flight per SM whatever the head_dim (a 4 x 2 CTA keeps 8
// blocks of K and V, 512 * head_dim bytes), since one SM's copies are
// latency-bound.  With one CTA per SM, 102400 tokens at head_dim 128 (32/8
// heads) streamed 5.1 TB/s and 131072 at head_dim 64 2.7 TB/s, against
// 6.3 TB/s at 256.  Registers and shared memory allow it: at head_dim 128 a
// CTA takes about 19K registers and 66 KB, at 64 about 14K and 34 KB.
int one_wave_ctas_per_sm(int head_dim) { return head_dim >= 256 ? 1 : head_dim >= 128 ? 2 : 4; }

int reduce_slice(int head_dim, long long pairs, int num_sms) {
    for (int w = head_dim; w > pa::kReduceMinSlice; w /= 2)
        if (pairs * (head_dim / w) >= 2ll * num_sms) return w;
    return pa::kReduceMinSlice;
}

int validate(const pa_decode_args* a, const pa_decode_opts* o) {
    if (!a) return PA_ERR_INVALID_ARG;
    if (a->num_seqs < 0 || a->num_seqs > 65535) return PA_ERR_INVALID_ARG;
    if (a->num_heads <= 0 || a->num_kv_heads <= 0 || a->head_dim <= 0 || a->block_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (a->num_heads % a->num_kv_heads) return PA_ERR_INVALID_ARG;
    if (!isfinite(a->scale)) return PA_ERR_INVALID_ARG;
    if (a->max_seq_len < 0 || a->max_blocks_per_seq < 0 || a->num_blocks < 0) return PA_ERR_INVALID_ARG;
    if (o && (o->mode < PA_MODE_AUTO || o->mode > PA_MODE_FLAT)) return PA_ERR_INVALID_ARG;
    if (o && o->partition_size < 0) return PA_ERR_INVALID_ARG;
    if (o && o->partition_size % a->block_size) return PA_ERR_INVALID_ARG;
    if (o && (o->warps < 0 || o->stages < 0)) return PA_ERR_INVALID_ARG;
    // every head_dim is compiled with the same set of CTA shapes; the
    // persistent kernel with one warp and 2 or 3 stages
    if (o && (o->mode == PA_MODE_PERSISTENT || o->mode == PA_MODE_FLAT)) {
        if ((o->warps || o->stages) &&
            pa::persistent_smem_bytes(256, o->warps ? o->warps : kPersistentWarps,
                                      o->stages ? o->stages : kPersistentStages) < 0)
            return PA_ERR_UNSUPPORTED;
        // the flat split keeps the batch's lengths and prefix sums in each CTA
        if (o->mode == PA_MODE_FLAT && a->num_seqs > pa::kPersistentSeqCache) return PA_ERR_UNSUPPORTED;
    } else if (o && (o->warps || o->stages) && pa::partition_smem_bytes(256, o->warps, o->stages) < 0) {
        return PA_ERR_UNSUPPORTED;
    }
    if (a->head_dim != 64 && a->head_dim != 128 && a->head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (a->block_size != pa::kBlockSize) return PA_ERR_UNSUPPORTED;
    if (a->num_heads / a->num_kv_heads > pa::kMaxGroup) return PA_ERR_UNSUPPORTED;
    // the grid must cover every sequence the block table can describe
    if ((long long)a->max_seq_len > (long long)a->max_blocks_per_seq * a->block_size) return PA_ERR_INVALID_ARG;
    // TMA row coordinates are 32-bit
    if (a->num_blocks * a->num_kv_heads * a->block_size >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
    if (a->num_seqs == 0) return PA_OK;
    if (!a->out || !a->q || !a->k_cache || !a->v_cache || !a->block_tables || !a->seq_lens) return PA_ERR_INVALID_ARG;
    if (!aligned(a->out, 16) || !aligned(a->q, 16) || !aligned(a->k_cache, 16) || !aligned(a->v_cache, 16) ||
        !aligned(a->block_tables, 4) || !aligned(a->seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (a->num_blocks == 0 && a->max_seq_len > 0) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

// Partition CTA shape (warps, stages per warp), picked with a wave model fitted
// to GB300 measurements.  A CTA keeps warps * stages blocks in flight, so on
// its own it streams at most that many bytes per HBM round trip (~1.6 us);
// the slots per SM follow from its shared memory; every wave of CTAs shares
// the HBM bandwidth and pays ~4 us of start-up and epilogue.  The shape with
// the smallest predicted time wins; ties go to more bytes in flight per CTA.
// The CTA count is exact for one sequence; for a batch, whose lengths the
// host does not see, half the grid is assumed (lengths spread up to the max).
struct CtaShape {
    int warps, stages;
};
constexpr CtaShape kShapes[] = {{2, 2}, {1, 2}, {1, 3}, {4, 2}};
constexpr double kHbmBytesPerUs = 6.8e6;
constexpr double kRoundTripUs = 1.6;
constexpr double kCtaOverheadUs = 4.0;
constexpr long long kSmemPerSm = 228 * 1024;

double predict_us(int head_dim, CtaShape sh, long long ctas, double bytes_per_cta, int num_sms) {
    const long long smem = pa::partition_smem_bytes(head_dim, sh.warps, sh.stages) + 1024;
    long long per_sm = kSmemPerSm / smem;
    if (per_sm > 2048 / (32 * sh.warps)) per_sm = 2048 / (32 * sh.warps);
    if (per_sm > 32) per_sm = 32;
    if (per_sm < 1) per_sm = 1;
    const long long slots = per_sm * num_sms;
    const double in_flight = (double)sh.warps * sh.stages * 2 * pa::kBlockSize * head_dim * 2;
    const double cta_rate = in_flight / kRoundTripUs;
    double t = 0;
    for (long long left = ctas; left > 0; left -= slots) {
        const long long k = left < slots ? left : slots;
        const double share = kHbmBytesPerUs / (double)k;
        t += bytes_per_cta / (share < cta_rate ? share : cta_rate) + kCtaOverheadUs;
    }
    return t;
}

void choose_shape(const pa_decode_args* a, const pa_decode_plan_t* plan, int num_sms, int* warps, int* stages) {
    // Batches of many (sequence, kv head) pairs of at most 16K tokens in the
    // default partitions: 2x2.  On ragged batches there the half-grid guess
    // below picks 1x3 or 1x2, measured 4-16 % slower than 2x2 (16 x U[1, 8192]
    // 65.9 -> 56.1 us, 48 x U[1, 4096] 80.2 -> 71.6, 100 x U[1, 1500] 63.4 ->
    // 56.4), while 2x2 stays within 2 % of the chosen shape elsewhere (uniform
    // batches, which do better still with PA_FLAG_UNIFORM_LENGTHS).
    if (plan->mode == PA_MODE_SPLIT && plan->partition_size == kDefaultPartition && a->num_seqs > 1 &&
        (long long)a->num_seqs * a->num_kv_heads >= kManyPairs && a->max_seq_len <= kManyPairsMaxLen &&
        a->head_dim >= 128) {
        *warps = 2;
        *stages = 2;
        return;
    }
    const long long grid = (long long)plan->grid_x * plan->grid_y * plan->grid_z;
    long long ctas = a->num_seqs == 1 ? grid : grid / 2;
    if (ctas < (long long)a->num_seqs * a->num_kv_heads) ctas = (long long)a->num_seqs * a->num_kv_heads;
    const int tokens = plan->partition_size < a->max_seq_len ? plan->partition_size : a->max_seq_len;
    const double bytes = (double)(tokens > 0 ? tokens : 1) * a->head_dim * 2 * 2;
    constexpr int n = (int)(sizeof(kShapes) / sizeof(kShapes[0]));
    double t[n], best = 0;
    for (int i = 0; i < n; ++i) {
        t[i] = predict_us(a->head_dim, kShapes[i], ctas, bytes, num_sms > 0 ? num_sms : 1);
        if (i == 0 || t[i] < best) best = t[i];
    }
    int pick = -1;
    for (int i = 0; i < n; ++i) {
        if (t[i] > best + 0.1) continue;
        const int fl = kShapes[i].warps * kShapes[i].stages;
        if (pick < 0 || fl > kShapes[pick].warps * kShapes[pick].stages ||
            (fl == kShapes[pick].warps * kShapes[pick].stages && kShapes[i].warps > kShapes[pick].warps))
            pick = i;
    }
    *warps = kShapes[pick].warps;
    *stages = kShapes[pick].stages;
}

// One-wave plans: 256 / head_dim 4-warp CTAs per SM (one_wave_ctas_per_sm),
// floor(SMs x that / (kv heads x sequences)) partitions per sequence of
// ceil(max_seq_len / that) tokens (whole blocks).  Device time per call on GB300 (4 kv heads, head_dim
// 256) against the grid of 512- or 256-token partitions:
//
// * Up to kOneWaveMinLen tokens (one round of copies for a 4-warp CTA)
//   SINGLE needs no reduce and wins (64 tokens: 3.6 us against 5.6).
//   Above it SINGLE adds about a microsecond per copy round (512 tokens:
//   8.55 -> 5.87 us, 400: 7.81 -> 5.86, 300: 6.54 -> 5.83, 200: 5.81 ->
//   5.67).
// * One sequence over kOneWaveMinLen tokens: its grid is known exactly.
//   Fewer, longer CTAs pay a CTA's start-up and merge once per SM and
//   leave fewer partials (102400 tokens 70.5 -> 68.9 us, 262144: 174.4 ->
//   161.6, 524288: 343.9 -> 305.0; 65536: 47.1 -> 45.5, 24000: 17.9 ->
//   14.1, 12000: 11.6 -> 9.7, 6000: 8.6 -> 8.3, 2048: 8.3 -> 6.5; the one
//   length measured slower was 8192, 8.8 -> 9.2).  From 2048-token
//   partitions on it is pooled (below); shorter ones measured no gain
//   from pooling (16384 tokens: 11.3 fixed, 13.7 pooled).
// * A batch whose partitions come to at most one round of copies
//   (kOneWaveShortMaxPartition tokens): every CTA ends after one round
//   whatever the lengths, so an uneven batch loses nothing the grid would
//   save (2 x 2048 8.72 -> 7.40, [2048, 40] 8.40 -> 7.40, 4 x 1024 9.27 ->
//   8.07, [1024, 50, 300, 700] 9.06 -> 7.80, 4 x 300 6.6 -> 6.0, 8 x 400
//   7.9 -> 6.8), when it gives at least kOneWaveShortMinParts partitions
//   per sequence of sequences over 256 tokens (SINGLE would need three
//   copy rounds or more).  Below that, SINGLE, with no reduce, won (8 x
//   256 5.89 against 6.29 us, 16 x 200 5.99 against 6.95, 12 x 300 6.65
//   against 7.40, 16 x 129 5.33 against 6.77); the reduce's cost grows
//   with the batch.
// * A batch whose sequences the caller states are all about max_seq_len
//   long (PA_FLAG_UNIFORM_LENGTHS), at any partition length (4 x 4096
//   14.5 -> 12.5 us, 4 x 16384 52.1 -> 46.0, 4 x 32768 85.7 -> 82.6, 2 x
//   65536 86.2 -> 82.4, 8 x 8192 51.7 -> 46.2, 16 x 16384 163.9 -> 158.4).
//   Without the statement the host cannot tell such a batch from one
//   whose longest sequence stands alone (4 x [32768, 100, 100, 100]: 30.8
//   -> 47.1 us) or whose lengths spread below the longest (8 x U[1, 8192]:
//   27.7 -> 37.7), so other batches keep the grid.
// Returns true and sets *part (and *pool) when the call takes a one-wave
// plan; the caller has left partition_size and the CTA shape to the library.
bool one_wave_partition(const pa_decode_args* a, const pa_decode_opts* o, int num_sms, int* part, bool* pool) {
    const int req_mode = o ? o->mode : PA_MODE_AUTO;
    if (a->num_seqs <= 0 || !(req_mode == PA_MODE_AUTO || req_mode == PA_MODE_SPLIT || req_mode == PA_MODE_FUSED))
        return false;
    // partitions of each sequence: one wave of 256 / head_dim CTAs per SM
    const long long per_seq =
        (long long)num_sms * one_wave_ctas_per_sm(a->head_dim) / ((long long)a->num_kv_heads * a->num_seqs);
    if (per_seq < 2) return false;
    const int bs = a->block_size;
    const long long p1 = ((a->max_seq_len + per_seq - 1) / per_seq + bs - 1) / bs * bs;
    const bool uniform = o && (o->flags & PA_FLAG_UNIFORM_LENGTHS);
    const bool one_seq = a->num_seqs == 1 && a->max_seq_len > kOneWaveMinLen;
    const bool stated = a->num_seqs > 1 && uniform;
    const bool short_seq = a->num_seqs > 1 && per_seq >= kOneWaveShortMinParts &&
                           a->max_seq_len > 2 * kOneWaveMinLen && p1 <= kOneWaveShortMaxPartition;
    if (!(one_seq || stated || short_seq)) return false;
    *part = static_cast<int>(p1);
    *pool = one_seq && p1 >= kOneWavePoolMinPartition;
    return true;
}

int make_plan(const pa_decode_args* a, const pa_decode_opts* o, int num_sms, pa_decode_plan_t* plan) {
    int rc = validate(a, o);
    if (rc) return rc;
    // The SM count only shapes the CTA choice and the reduce grid; without a
    // device the launch reports the error later, so a failed query plans for one SM.
    if (num_sms <= 0 && query_sm_count(&num_sms) != PA_OK) num_sms = 1;
    memset(plan, 0, sizeof(*plan));
    const int bs = a->block_size;
    int part = (o && o->partition_size > 0) ? o->partition_size : kDefaultPartition;
    if (!(o && o->partition_size > 0) && a->max_seq_len > kDefaultPartition) {
        // Short work: when partitions of the default size would give fewer CTAs
        // than SMs, halve them so that twice as many SMs stream the cache (an
        // early measurement on 2048 tokens, which now take a one-wave plan:
        // 13.7 -> 10.5 us; smaller partitions cost more in the reduce).
        const long long ctas = (long long)((a->max_seq_len + kDefaultPartition - 1) / kDefaultPartition) *
                               a->num_kv_heads * a->num_seqs;
        if (ctas < num_sms) part = kDefaultPartition / 2;
    }
    // one-wave plans (see one_wave_partition)
    bool one_wave = false, pool_one_wave = false;
    if (!(o && o->partition_size > 0) && !(o && (o->warps || o->stages)))
        one_wave = one_wave_partition(a, o, num_sms, &part, &pool_one_wave);
    const int split_parts = (a->max_seq_len + part - 1) / part;
    int mode = o ? o->mode : PA_MODE_AUTO;
    if (mode == PA_MODE_AUTO) {
        // A sequence that fits one partition needs no reduce.  Otherwise split:
        // with few (sequence, kv head) pairs a single-pass grid leaves most of
        // the SMs idle, and with many its time is set by the longest sequence.
        mode = split_parts <= 1 ? PA_MODE_SINGLE : PA_MODE_SPLIT;
    }
    plan->mode = mode;
    if (mode == PA_MODE_SINGLE) {
        const int whole = ((a->max_seq_len + bs - 1) / bs) * bs;
        plan->partition_size = whole > 0 ? whole : bs;
        plan->grid_x = 1;
    } else {
        plan->partition_size = part;
        plan->grid_x = split_parts > 0 ? split_parts : 1;
    }
    plan->max_partitions = plan->grid_x;
    plan->grid_y = a->num_kv_heads;
    plan->grid_z = a->num_seqs;
    int warps = o ? o->warps : 0, stages = o ? o->stages : 0;
    const bool apportion = mode == PA_MODE_PERSISTENT && !(o && o->partition_size > 0);
    const bool flat = mode == PA_MODE_FLAT;
    if (mode == PA_MODE_PERSISTENT || flat) {
        if (!warps) warps = (apportion || flat) ? kPersistentWarps : kPersistentWarpsFixedSize;
        if (!stages) stages = kPersistentStages;
    } else if (one_wave) {
        warps = 4;
        stages = 2;
    } else if (!warps) {
        choose_shape(a, plan, num_sms, &warps, &stages);
    }
    plan->threads = warps * 32;
    plan->stages = stages;
    plan->smem_bytes = (mode == PA_MODE_PERSISTENT || flat) ? pa::persistent_smem_bytes(a->head_dim, warps, stages) +
                                                                  pa::persistent_seq_cache_bytes(a->num_seqs)
                                                            : pa::partition_smem_bytes(a->head_dim, warps, stages);
    if (flat) {
        // one wave (one CTA per SM at head_dim 256, more below it, as for the
        // one-wave plans): C CTAs per kv head, each streaming an equal share
        // of the batch's blocks (the share is fixed on the device)
        const int slots = num_sms * one_wave_ctas_per_sm(a->head_dim);
        const int C = slots / a->num_kv_heads > 0 ? slots / a->num_kv_heads : 1;
        plan->grid_x = C * a->num_kv_heads;
        plan->grid_y = plan->grid_z = 1;
        plan->partition_size = 0;
        plan->max_partitions = C;
    }
    if (mode == PA_MODE_PERSISTENT) {
        // a fixed grid of every CTA the SMs hold at once
        long long per_sm = kSmemPerSm / (plan->smem_bytes + 1024);
        if (per_sm > 2048 / plan->threads) per_sm = 2048 / plan->threads;
        if (per_sm > 32) per_sm = 32;
        if (per_sm < 1) per_sm = 1;
        plan->grid_x = (int)(per_sm * num_sms);
        plan->grid_y = plan->grid_z = 1;
        if (apportion) {
            // partitions per kv head shared out over the batch: about one wave
            plan->partition_size = 0;
            plan->max_partitions = plan->grid_x / a->num_kv_heads > 1 ? plan->grid_x / a->num_kv_heads : 1;
        }
        // the work list holds at most num_seqs * (max_partitions + 1) * num_kv_heads items
        if ((long long)a->num_seqs * (plan->max_partitions + 1) * a->num_kv_heads >= (1ll << 31))
            return PA_ERR_UNSUPPORTED;
    }
    plan->launch_reduce =
        ((mode == PA_MODE_SPLIT || mode == PA_MODE_PERSISTENT || flat) && plan->max_partitions > 1) ? 1 : 0;
    // FUSED on a grid the device holds at once merges in parallel after a
    // group barrier (a cooperative launch), when the staged slice of the
    // merge fits the CTA's stage area; otherwise the last CTA of a group merges
    if (mode == PA_MODE_FUSED && plan->grid_x > 1) {
        long long per_sm = kSmemPerSm / (plan->smem_bytes + 1024);
        if (per_sm > 2048 / plan->threads) per_sm = 2048 / plan->threads;
        if (per_sm > 32) per_sm = 32;
        const long long ctas = (long long)plan->grid_x * plan->grid_y * plan->grid_z;
        const long long stage_area = (long long)warps * stages * 2 * pa::kBlockSize * a->head_dim * 2;
        plan->coop = ctas <= per_sm * num_sms &&
                     pa::fused_barrier_bytes(plan->grid_x, a->num_heads / a->num_kv_heads, a->head_dim) <= stage_area;
    }
    // Pooled: on request, and by default for the one-wave plan of one long
    // sequence (short ones measured no gain: 4096 tokens 7.61 -> 7.54 us,
    // 2048 6.48 -> 6.50), where every CTA is resident from the start and the SMs'
    // unequal shares of HBM bandwidth would otherwise set the finish (GB300,
    // 102400 tokens: 66.8 -> 65.4 us per call; 262144: 158.5 -> 156.0).  The
    // one-wave plan of a uniform batch stays fixed (pooled: 4 x 32768 82.6 ->
    // 81.8 us, 2 x 65536 82.4 -> 83.1).  Plans of several waves stay fixed: a
    // later wave's CTAs would find only their first chunks left.
    const int flags = o ? o->flags : 0;
    const bool want_pool =
        (flags & PA_FLAG_POOLED) || (pool_one_wave && !(flags & PA_FLAG_DETERMINISTIC));
    // (the claim counters are re-armed by the reduce kernel, or by the last
    // CTA to leave a fused group's barrier)
    plan->pooled = want_pool && !(flags & PA_FLAG_DETERMINISTIC) &&
                   ((mode == PA_MODE_SPLIT && plan->launch_reduce) || (mode == PA_MODE_FUSED && plan->coop)) &&
                   plan->partition_size >= pa::pool_min_partition(warps, stages);
    if (mode == PA_MODE_FUSED)
        plan->workspace_bytes =
            fused_workspace_bytes(a->num_seqs, a->num_heads, a->num_kv_heads, plan->grid_x, a->head_dim);
    if (plan->launch_reduce) {
        plan->reduce_grid_x = a->num_heads;
        plan->reduce_grid_y = a->num_seqs;
        plan->reduce_grid_z = a->head_dim / reduce_slice(a->head_dim, (long long)a->num_seqs * a->num_heads, num_sms);
        plan->workspace_bytes = split_workspace_bytes(a->num_seqs, a->num_heads, plan->max_partitions, a->head_dim);
    }
    if (plan->pooled && mode == PA_MODE_SPLIT)  // + the claim counters (inside FUSED's layout already)
        plan->workspace_bytes += claims_bytes(a->num_seqs, a->num_kv_heads);
    if (mode == PA_MODE_PERSISTENT)  // + the work list and item counter, the order, the partition sizes
        plan->workspace_bytes = split_workspace_bytes(a->num_seqs, a->num_heads, plan->max_partitions, a->head_dim) +
                                align_up(static_cast<size_t>(a->num_seqs + 2) * 4, kWsAlign) +
                                2 * align_up(static_cast<size_t>(a->num_seqs) * 4, kWsAlign);
    if (flat)  // + each sequence's number of partials
        plan->workspace_bytes = split_workspace_bytes(a->num_seqs, a->num_heads, plan->max_partitions, a->head_dim) +
                                align_up(static_cast<size_t>(a->num_seqs) * 4, kWsAlign);
    return PA_OK;
}

// cuTensorMapEncodeTiled, reached through the runtime so the library needs no
// link-time dependency on the driver (it still loads on machines without one).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// A cache viewed as a 2-D tensor of (num_blocks * num_kv_heads * block_size)
// rows by head_dim halves; a box is block_size rows by 64 halves (128 bytes),
// stored with the 128-byte swizzle.  Rows past the pool read as zero.
int make_cache_map(CUtensorMap* map, const void* base, const pa_decode_args* a) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PA_ERR_CUDA;
    const cuuint64_t rows = static_cast<cuuint64_t>(a->num_blocks) * a->num_kv_heads * a->block_size;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a->head_dim), rows > 0 ? rows : 1};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a->head_dim) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(a->block_size)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int make_cache_block_map(CUtensorMap* map, const void* base, long long num_blocks, int num_kv_heads, int head_dim);

// Diagnostic builds (-DPA_TRACE): device buffer for per-CTA timestamps of
// the partition kernel (5 x 8 bytes per CTA) or of the tcgen05 prefix kernel
// (kPrefixTraceIters x 16 x 8 bytes per CTA), set by pa_debug_set_trace.
unsigned long long* g_trace = nullptr;

int run(const pa_decode_args* a, const pa_decode_opts* o, void* ws, size_t ws_bytes, cudaStream_t stream,
        const pa_decode_plan_t& plan) {
    if (a->num_seqs == 0) return PA_OK;
    if (plan.workspace_bytes > 0 && (!ws || ws_bytes < plan.workspace_bytes || !aligned(ws, kWsAlign)))
        return PA_ERR_WORKSPACE;

    CUtensorMap tk, tv;
    int rc = make_cache_block_map(&tk, a->k_cache, a->num_blocks, a->num_kv_heads, a->head_dim);
    if (rc) return rc;
    rc = make_cache_block_map(&tv, a->v_cache, a->num_blocks, a->num_kv_heads, a->head_dim);
    if (rc) return rc;

    const size_t rows = static_cast<size_t>(a->num_seqs) * a->num_heads * plan.max_partitions;
    uint8_t* w = static_cast<uint8_t*>(ws);
    pa::PartitionParams prm;
    prm.out = static_cast<__half*>(a->out);
    prm.q = static_cast<const __half*>(a->q);
    prm.block_tables = a->block_tables;
    prm.seq_lens = a->seq_lens;
    const bool fused = plan.mode == PA_MODE_FUSED && plan.grid_x > 1;
    const bool flat = plan.mode == PA_MODE_FLAT;
    const bool persistent = plan.mode == PA_MODE_PERSISTENT || flat;
    const bool partials = plan.launch_reduce || fused;
    const size_t partial_bytes = split_workspace_bytes(a->num_seqs, a->num_heads, plan.max_partitions, a->head_dim);
    prm.max_logits = partials ? reinterpret_cast<float*>(w) : nullptr;
    prm.exp_sums = partials ? reinterpret_cast<float*>(w + align_up(rows * 4, kWsAlign)) : nullptr;
    prm.tmp_out = partials ? reinterpret_cast<float*>(w + 2 * align_up(rows * 4, kWsAlign)) : nullptr;
    prm.tickets = fused ? reinterpret_cast<unsigned int*>(w + partial_bytes + claims_bytes(a->num_seqs, a->num_kv_heads))
                        : nullptr;
    prm.claims = plan.pooled ? reinterpret_cast<unsigned long long*>(w + partial_bytes) : nullptr;
    // persistent schedule tables after the partials: work list + counter, order, partition sizes
    // (the flat split: each sequence's number of partials)
    const bool listed = persistent && !flat;
    int* list = listed ? reinterpret_cast<int*>(w + partial_bytes) : nullptr;
    int* order = listed ? reinterpret_cast<int*>(w + partial_bytes +
                                                 align_up(static_cast<size_t>(a->num_seqs + 2) * 4, kWsAlign))
                        : nullptr;
    int* parts = listed ? order + align_up(static_cast<size_t>(a->num_seqs) * 4, kWsAlign) / 4 : nullptr;
    prm.flat = flat ? 1 : 0;
    prm.part_counts = flat && plan.launch_reduce ? reinterpret_cast<int*>(w + partial_bytes) : nullptr;
    prm.work_offsets = list;
    prm.work_counter = listed ? list + a->num_seqs + 1 : nullptr;
    prm.seq_order = order;
    prm.part_sizes = parts;
    prm.num_seqs = a->num_seqs;
    prm.status = persistent ? pa::device_status_ptr() : nullptr;
    if (persistent && !prm.status) return PA_ERR_CUDA;
    prm.num_blocks = a->num_blocks;
    prm.num_heads = a->num_heads;
    prm.num_kv_heads = a->num_kv_heads;
    prm.group = a->num_heads / a->num_kv_heads;
    prm.max_blocks_per_seq = a->max_blocks_per_seq;
    prm.max_seq_len = a->max_seq_len;
    prm.partition_size = plan.partition_size;
    prm.max_partitions = plan.max_partitions;
    prm.scale_log2 = static_cast<float>(static_cast<double>(a->scale) * 1.4426950408889634);
    prm.wait_limit = (o && o->wait_limit) ? o->wait_limit : pa::kDefaultWaitLimit;
    prm.force_timeout = (o && (o->flags & PA_FLAG_FORCE_TIMEOUT)) ? 1 : 0;
    prm.trace = g_trace;
    prm.coop = fused && plan.coop ? 1 : 0;

    if (listed) {
        pa::ScanParams sp;
        sp.seq_lens = a->seq_lens;
        sp.work_offsets = list;
        sp.seq_order = order;
        sp.part_sizes = parts;
        sp.work_counter = list + a->num_seqs + 1;
        sp.num_seqs = a->num_seqs;
        sp.max_seq_len = a->max_seq_len;
        sp.max_blocks_per_seq = a->max_blocks_per_seq;
        sp.num_kv_heads = a->num_kv_heads;
        sp.first_dynamic = plan.grid_x;
        sp.partition_size = plan.partition_size;  // 0: apportion max_partitions per kv head
        sp.slots = plan.max_partitions;
        if (pa::launch_work_scan(sp, stream) != cudaSuccess) return PA_ERR_CUDA;
    }
    if (o && o->event_partition_begin &&
        cudaEventRecord(static_cast<cudaEvent_t>(o->event_partition_begin), stream) != cudaSuccess)
        return PA_ERR_CUDA;
    cudaError_t le =
        persistent ? pa::launch_partition_persistent(a->head_dim, plan.threads / 32, plan.stages, prm, tk, tv,
                                                     plan.grid_x, stream)
                   : pa::launch_partition(a->head_dim, plan.threads / 32, plan.stages, prm, tk, tv,
                                          dim3(plan.grid_x, plan.grid_y, plan.grid_z), stream);
    if (le == cudaErrorCooperativeLaunchTooLarge && prm.coop) {
        // the device holds fewer CTAs at once than the plan assumed: the last
        // CTA of each group merges instead, with fixed partitions
        cudaGetLastError();
        prm.coop = 0;
        prm.claims = nullptr;
        le = pa::launch_partition(a->head_dim, plan.threads / 32, plan.stages, prm, tk, tv,
                                  dim3(plan.grid_x, plan.grid_y, plan.grid_z), stream);
    }
    if (le != cudaSuccess) return PA_ERR_CUDA;
    if (o && o->event_partition_end &&
        cudaEventRecord(static_cast<cudaEvent_t>(o->event_partition_end), stream) != cudaSuccess)
        return PA_ERR_CUDA;
    if (plan.launch_reduce) {
        pa::ReduceParams rp;
        rp.out = prm.out;
        rp.max_logits = prm.max_logits;
        rp.exp_sums = prm.exp_sums;
        rp.tmp_out = prm.tmp_out;
        rp.seq_lens = a->seq_lens;
        rp.num_heads = a->num_heads;
        rp.max_blocks_per_seq = a->max_blocks_per_seq;
        rp.max_seq_len = a->max_seq_len;
        rp.partition_size = plan.partition_size;
        rp.max_partitions = plan.max_partitions;
        rp.part_sizes = parts;
        rp.part_counts = prm.part_counts;
        rp.claims = prm.claims;
        rp.group = prm.group;
        if (pa::launch_reduce(a->head_dim, a->head_dim / plan.reduce_grid_z, rp,
                              dim3(plan.reduce_grid_x, plan.reduce_grid_y, plan.reduce_grid_z), stream) != cudaSuccess) {
            // The partition grid may have consumed claims, and only the reduce
            // re-arms the counters: disarm them, so the next pooled call on this
            // workspace deals its chunks round-robin instead of skipping some.
            if (prm.claims) pa::disarm_claims(prm.claims, static_cast<size_t>(a->num_seqs) * a->num_kv_heads, stream);
            return PA_ERR_CUDA;
        }
    }
    return PA_OK;
}

// Partials of partitions [begin, begin + count) of every sequence, into the
// caller's arrays (split-KV across devices: each device computes its own range
// of partitions over its own part of the cache; pa_merge_partials merges them).
int run_partials(const pa_decode_args* a, const pa_decode_opts* o, int partition_size, int begin, int count,
                 float* max_logits, float* exp_sums, float* tmp_out, cudaStream_t stream) {
    if (!a) return PA_ERR_INVALID_ARG;
    if (partition_size <= 0 || begin < 0 || count <= 0) return PA_ERR_INVALID_ARG;
    if ((long long)(begin + (long long)count) * partition_size >= (1ll << 31)) return PA_ERR_INVALID_ARG;
    if (o && o->mode != PA_MODE_AUTO && o->mode != PA_MODE_SPLIT) return PA_ERR_INVALID_ARG;
    pa_decode_args ca = *a;
    ca.out = tmp_out;  // the output is never written; the partials take its place
    pa_decode_opts co;
    memset(&co, 0, sizeof(co));
    if (o) co = *o;
    co.mode = PA_MODE_SPLIT;
    co.partition_size = partition_size;
    co.flags = (co.flags & PA_FLAG_FORCE_TIMEOUT) | PA_FLAG_DETERMINISTIC;  // fixed partitions, never pooled
    pa_decode_plan_t plan;
    int rc = make_plan(&ca, &co, 0, &plan);
    if (rc) return rc;
    if (a->num_seqs == 0) return PA_OK;
    if (!max_logits || !exp_sums || !tmp_out || !aligned(max_logits, 4) || !aligned(exp_sums, 4) ||
        !aligned(tmp_out, 16))
        return PA_ERR_INVALID_ARG;
    plan.grid_x = count;
    plan.max_partitions = count;
    if (!co.warps && !co.stages) {
        int num_sms = 0;
        if (query_sm_count(&num_sms) != PA_OK) num_sms = 1;
        int warps = 0, stages = 0;
        choose_shape(&ca, &plan, num_sms, &warps, &stages);
        plan.threads = warps * 32;
        plan.stages = stages;
    }

    CUtensorMap tk, tv;
    if ((rc = make_cache_block_map(&tk, a->k_cache, a->num_blocks, a->num_kv_heads, a->head_dim)) ||
        (rc = make_cache_block_map(&tv, a->v_cache, a->num_blocks, a->num_kv_heads, a->head_dim)))
        return rc;
    pa::PartitionParams prm{};
    prm.out = nullptr;
    prm.q = static_cast<const __half*>(a->q);
    prm.block_tables = a->block_tables;
    prm.seq_lens = a->seq_lens;
    prm.max_logits = max_logits;
    prm.exp_sums = exp_sums;
    prm.tmp_out = tmp_out;
    prm.num_seqs = a->num_seqs;
    prm.num_blocks = a->num_blocks;
    prm.num_heads = a->num_heads;
    prm.num_kv_heads = a->num_kv_heads;
    prm.group = a->num_heads / a->num_kv_heads;
    prm.max_blocks_per_seq = a->max_blocks_per_seq;
    prm.max_seq_len = a->max_seq_len;
    prm.partition_size = partition_size;
    prm.max_partitions = count;
    prm.scale_log2 = static_cast<float>(static_cast<double>(a->scale) * 1.4426950408889634);
    prm.wait_limit = co.wait_limit ? co.wait_limit : pa::kDefaultWaitLimit;
    prm.force_timeout = (co.flags & PA_FLAG_FORCE_TIMEOUT) ? 1 : 0;
    prm.trace = g_trace;
    prm.part_begin = begin;
    prm.partials_only = 1;
    if (co.event_partition_begin &&
        cudaEventRecord(static_cast<cudaEvent_t>(co.event_partition_begin), stream) != cudaSuccess)
        return PA_ERR_CUDA;
    if (pa::launch_partition(a->head_dim, plan.threads / 32, plan.stages, prm, tk, tv,
                             dim3(plan.grid_x, plan.grid_y, plan.grid_z), stream) != cudaSuccess)
        return PA_ERR_CUDA;
    if (co.event_partition_end &&
        cudaEventRecord(static_cast<cudaEvent_t>(co.event_partition_end), stream) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

// The log-sum-exp merge of partials gathered from num_sources sources, each
// holding partitions_per_source consecutive partitions of every sequence.
int run_merge(void* out, const float* max_logits, const float* exp_sums, const float* tmp_out,
              const int32_t* seq_lens, int num_seqs, int num_heads, int head_dim, int max_seq_len, int partition_size,
              int num_sources, int partitions_per_source, cudaStream_t stream) {
    if (num_seqs < 0 || num_seqs > 65535 || num_heads <= 0 || max_seq_len < 0) return PA_ERR_INVALID_ARG;
    if (partition_size <= 0 || partition_size % pa::kBlockSize || num_sources <= 0 || partitions_per_source <= 0)
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
    const long long slots = (long long)num_sources * partitions_per_source;
    if (slots >= (1ll << 31)) return PA_ERR_INVALID_ARG;
    // the sources must cover every partition of the longest sequence
    if ((max_seq_len + (long long)partition_size - 1) / partition_size > slots) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !max_logits || !exp_sums || !tmp_out || !seq_lens || !aligned(out, 16) || !aligned(tmp_out, 16) ||
        !aligned(max_logits, 4) || !aligned(exp_sums, 4) || !aligned(seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    int num_sms = 0;
    if (query_sm_count(&num_sms) != PA_OK) num_sms = 1;
    pa::ReduceParams rp{};
    rp.out = static_cast<__half*>(out);
    rp.max_logits = max_logits;
    rp.exp_sums = exp_sums;
    rp.tmp_out = tmp_out;
    rp.seq_lens = seq_lens;
    rp.num_heads = num_heads;
    rp.max_seq_len = max_seq_len;
    rp.max_blocks_per_seq = (max_seq_len + pa::kBlockSize - 1) / pa::kBlockSize;
    rp.partition_size = partition_size;
    rp.max_partitions = static_cast<int>(slots);
    rp.part_sizes = nullptr;
    rp.claims = nullptr;
    rp.group = 1;
    rp.src_parts = partitions_per_source;
    rp.src_stride = (long long)num_seqs * num_heads * partitions_per_source;
    const int width = reduce_slice(head_dim, (long long)num_seqs * num_heads, num_sms);
    return pa::launch_reduce(head_dim, width, rp, dim3(num_heads, num_seqs, head_dim / width), stream) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

// New tokens' K or V viewed as a 3-D tensor [num_tokens][num_kv_heads][head_dim];
// a box is 16 tokens x 1 kv head x 64 halves with the 128-byte swizzle, the
// same shared-memory layout as a cache box.  Tokens past the end read as zero.
int make_new_kv_map(CUtensorMap* map, const void* base, int num_tokens, int num_kv_heads, int head_dim) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PA_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_kv_heads, (cuuint64_t)(num_tokens > 0 ? num_tokens : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_kv_heads * head_dim * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)pa::kBlockSize};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// Whole-block views: one box brings a block's 16 rows x head_dim as
// [64-column chunk][16 rows][128 B] (each chunk with the 128-byte swizzle),
// the stage layout of the decode kernels and of the tcgen05 prefix kernel's
// P.V operand.  A TMA instruction holds its issuing thread for a fixed time
// whatever the box size, so one box per tile instead of one per 64-column
// chunk cuts that time by D / 64.  Cache: dims (64 halves, rows, chunk), the
// chunk dimension stepping 128 B through a row.
int make_cache_block_map(CUtensorMap* map, const void* base, long long num_blocks, int num_kv_heads, int head_dim) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PA_ERR_CUDA;
    const cuuint64_t rows = static_cast<cuuint64_t>(num_blocks) * num_kv_heads * pa::kBlockSize;
    cuuint64_t dims[3] = {64, rows > 0 ? rows : 1, static_cast<cuuint64_t>(head_dim / 64)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2, 128};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(pa::kBlockSize), static_cast<cuuint32_t>(head_dim / 64)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// The same for the chunk's packed [token][kv head][head_dim] tensor: dims
// (64 halves, kv head, token, chunk); tokens past the tensor read as zeros.
int make_new_kv_block_map(CUtensorMap* map, const void* base, int num_tokens, int num_kv_heads, int head_dim) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PA_ERR_CUDA;
    cuuint64_t dims[4] = {64, (cuuint64_t)num_kv_heads, (cuuint64_t)(num_tokens > 0 ? num_tokens : 1),
                          (cuuint64_t)(head_dim / 64)};
    cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_kv_heads * head_dim * 2, 128};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)pa::kBlockSize, (cuuint32_t)(head_dim / 64)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int validate_prefix(const pa_prefix_args* a, const pa_decode_opts* o) {
    if (!a) return PA_ERR_INVALID_ARG;
    if (a->num_seqs < 0 || a->num_seqs > 65535 || a->num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (a->num_heads <= 0 || a->num_kv_heads <= 0 || a->head_dim <= 0 || a->block_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (a->num_heads % a->num_kv_heads) return PA_ERR_INVALID_ARG;
    if (!isfinite(a->scale)) return PA_ERR_INVALID_ARG;
    if (a->max_context_len < 0 || a->max_query_len < 0 || a->max_blocks_per_seq < 0 || a->num_blocks < 0)
        return PA_ERR_INVALID_ARG;
    if (o && (o->mode < PA_MODE_AUTO || o->mode > PA_MODE_SPLIT)) return PA_ERR_INVALID_ARG;
    if (a->head_dim != 64 && a->head_dim != 128 && a->head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (a->block_size != pa::kBlockSize) return PA_ERR_UNSUPPORTED;
    if (a->num_heads / a->num_kv_heads > pa::kMaxGroup) return PA_ERR_UNSUPPORTED;
    if ((long long)a->max_context_len > (long long)a->max_blocks_per_seq * a->block_size) return PA_ERR_INVALID_ARG;
    if (a->num_blocks * a->num_kv_heads * a->block_size >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
    if (a->num_tokens > 0 && a->max_query_len == 0) return PA_ERR_INVALID_ARG;
    // the kernels number their units (query tiles x kv heads x sequences,
    // tiles of at least 128 / G tokens) in 32 bits
    const long long tile_tokens = 128 / (a->num_heads / a->num_kv_heads);
    if ((a->max_query_len + tile_tokens - 1) / tile_tokens * a->num_kv_heads * a->num_seqs >= (1ll << 31))
        return PA_ERR_UNSUPPORTED;
    if (a->num_seqs == 0 || a->num_tokens == 0) return PA_OK;
    if (!a->out || !a->q || !a->k_new || !a->v_new || !a->k_cache || !a->v_cache || !a->block_tables ||
        !a->context_lens || !a->query_start_loc)
        return PA_ERR_INVALID_ARG;
    if (!aligned(a->out, 16) || !aligned(a->q, 16) || !aligned(a->k_new, 16) || !aligned(a->v_new, 16) ||
        !aligned(a->k_cache, 16) || !aligned(a->v_cache, 16) || !aligned(a->block_tables, 4) ||
        !aligned(a->context_lens, 4) || !aligned(a->query_start_loc, 4))
        return PA_ERR_INVALID_ARG;
    if (a->num_blocks == 0 && a->max_context_len > 0) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

// Key split of the tensor-core prefill kernel's last round (pa_prefix_split).
// Every CTA of that kernel walks all keys of its sequence, so with one CTA
// per SM a grid of N CTAs on S SMs takes about ceil(N / S) rounds of T.  When
// the last round holds R = N mod S CTAs, splitting those R tiles into k key
// ranges gives R k CTAs of about (T - f) / k + f each, in ceil(R k / S)
// rounds, plus a merge.  T = f + tiles * t_tile with f ~ 7 us of fixed cost
// per CTA and t_tile ~ 0.9 us per 64-key tile (GB300, head_dim 256; per-CTA
// phase traces), tiles from the longest context and chunk.  The k in [2, 8]
// with the shortest last rounds is taken if it saves at least 5 % of T.  On
// 4 x 8192 cached tokens with chunks of 512 (400 CTAs, 96 in the last round)
// the model takes k = 3, the fastest of the measured splits (us per call:
// none 381.6, k = 3 373.1, k = 2 401.2, k = 4 385.2, k = 5 400.5, k = 6 394.2;
// the last 248 tiles in 3: 410.8; every tile in 2: 453.4): a part costs more
// than (T - f) / k + f, since it also writes its rows in fp32 for the merge.
struct PrefixSplit {
    int parts = 0, whole = 0, units = 0, tiles_per_seq = 0;
};

constexpr double kPrefixFixedUs = 7.0, kPrefixTileUs = 0.9, kPrefixMergeUs = 3.0;
constexpr long long kPrefixSplitMaxRounds = 4;

int plan_prefix_split(const pa_prefix_args* a, const pa_prefix_split_opts* split, int num_sms, PrefixSplit* sp) {
    *sp = PrefixSplit{};
    const int tile_tokens = pa::kPrefixTileRows / (a->num_heads / a->num_kv_heads);
    sp->tiles_per_seq = (a->max_query_len + tile_tokens - 1) / tile_tokens;
    const long long n = (long long)sp->tiles_per_seq * a->num_kv_heads * a->num_seqs;
    if (split && split->parts != 0) {
        if (split->parts < 1 || split->parts > 64 || split->units < 0 || split->units > n) return PA_ERR_INVALID_ARG;
        if ((long long)split->units * split->parts + (n - split->units) >= (1ll << 31)) return PA_ERR_INVALID_ARG;
        if (split->units == 0) return PA_OK;
        sp->parts = split->parts;
        sp->units = split->units;
        sp->whole = static_cast<int>(n - split->units);
        return PA_OK;
    }
    // Only a grid of a few rounds has a clean partial last round: with more,
    // the CTAs of a ragged batch differ in length and already fill it (the
    // 16-sequence mixed batch, 21 rounds: 528 -> 542 us when split).
    if (num_sms <= 0 || n <= num_sms || n > kPrefixSplitMaxRounds * num_sms) return PA_OK;
    const long long r = n % num_sms;
    if (r == 0) return PA_OK;
    const long long tiles = ((a->max_context_len + pa::kBlockSize - 1) / pa::kBlockSize +
                             (a->max_query_len + pa::kBlockSize - 1) / pa::kBlockSize + 3) / 4;
    const double t = kPrefixFixedUs + tiles * kPrefixTileUs;
    double best = t;  // the last round of whole tiles
    int best_k = 0;
    for (int k = 2; k <= 8; ++k) {
        const long long rounds = (r * k + num_sms - 1) / num_sms;
        const double tk = rounds * ((t - kPrefixFixedUs) / k + kPrefixFixedUs) + kPrefixMergeUs;
        if (tk < best) {
            best = tk;
            best_k = k;
        }
    }
    if (best_k == 0 || best > 0.95 * t) return PA_OK;
    sp->parts = best_k;
    sp->units = static_cast<int>(r);
    sp->whole = static_cast<int>(n - r);
    return PA_OK;
}

size_t prefix_split_o_bytes(const PrefixSplit& sp, int head_dim) {
    return align_up((size_t)sp.units * sp.parts * pa::kPrefixTileRows * head_dim * 4, kWsAlign);
}

size_t prefix_split_bytes(const PrefixSplit& sp, int head_dim) {
    if (!sp.parts) return 0;
    return prefix_split_o_bytes(sp, head_dim) +
           align_up((size_t)sp.units * sp.parts * pa::kPrefixTileRows * 2 * 4, kWsAlign);
}

// The persistent prefill's claim counter and finish count, one pair per
// (device, stream), zeroed on the stream when first used; each call's last
// CTA re-arms them.  Calls on one stream never overlap, so no two running
// grids share a pair.
std::mutex g_sched_mutex;
std::map<std::pair<int, uintptr_t>, unsigned int*> g_sched;

bool prefix_sched_ready(cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(g_sched_mutex);
    return g_sched.count({dev, reinterpret_cast<uintptr_t>(stream)}) != 0;
}

int ensure_prefix_sched(cudaStream_t stream, unsigned int** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_sched_mutex);
    const auto key = std::make_pair(dev, reinterpret_cast<uintptr_t>(stream));
    auto it = g_sched.find(key);
    if (it == g_sched.end()) {
        void* p = nullptr;
        if (cudaMalloc(&p, 256) != cudaSuccess) {
            cudaGetLastError();
            return PA_ERR_OOM;
        }
        if (cudaMemsetAsync(p, 0, 256, stream) != cudaSuccess) {
            cudaFree(p);
            return PA_ERR_CUDA;
        }
        it = g_sched.emplace(key, static_cast<unsigned int*>(p)).first;
    }
    *out = it->second;
    return PA_OK;
}

// split_call: pa_prefix_split (the key split of `split`, or the plan's,
// into workspace `ws`); otherwise pa_prefix / pa_prefix_ex.
int run_prefix(const pa_prefix_args* a, const pa_decode_opts* o, cudaStream_t stream, bool split_call = false,
               const pa_prefix_split_opts* split = nullptr, void* ws = nullptr, size_t ws_bytes = 0) {
    int rc = validate_prefix(a, o);
    if (rc) return rc;
    if (a->num_seqs == 0 || a->num_tokens == 0) return PA_OK;
    pa_decode_args ca;  // the cache part, for the shared tensor-map helper
    memset(&ca, 0, sizeof(ca));
    ca.num_blocks = a->num_blocks > 0 ? a->num_blocks : 1;
    ca.num_kv_heads = a->num_kv_heads;
    ca.head_dim = a->head_dim;
    ca.block_size = a->block_size;
    // tensor-core (tcgen05) kernel by default; the warp-level MMA kernel on request
    const bool warp_mma = o && (o->flags & PA_FLAG_PREFIX_WARP_MMA);
    // the key split and its workspace are checked before any CUDA call but
    // the SM count (which only the library's own plan reads)
    PrefixSplit sp;
    if (split_call && !warp_mma) {
        int num_sms = 0;
        if (!(split && split->parts) && query_sm_count(&num_sms) != PA_OK) return PA_ERR_CUDA;
        if ((rc = plan_prefix_split(a, split, num_sms, &sp))) return rc;
        if (sp.parts && (!ws || ws_bytes < prefix_split_bytes(sp, a->head_dim) || !aligned(ws, kWsAlign)))
            return PA_ERR_INVALID_ARG;
    }
    // K cache, V cache, K new, V new; the tcgen05 kernel copies V a whole block per box
    CUtensorMap maps[4];
    if ((rc = make_cache_map(&maps[0], a->k_cache, &ca)) ||
        (rc = make_new_kv_map(&maps[2], a->k_new, a->num_tokens, a->num_kv_heads, a->head_dim)))
        return rc;
    if (warp_mma) {
        if ((rc = make_cache_map(&maps[1], a->v_cache, &ca)) ||
            (rc = make_new_kv_map(&maps[3], a->v_new, a->num_tokens, a->num_kv_heads, a->head_dim)))
            return rc;
    } else if ((rc = make_cache_block_map(&maps[1], a->v_cache, ca.num_blocks, a->num_kv_heads, a->head_dim)) ||
               (rc = make_new_kv_block_map(&maps[3], a->v_new, a->num_tokens, a->num_kv_heads, a->head_dim))) {
        return rc;
    }
    pa::PrefixParams prm;
    prm.out = static_cast<__half*>(a->out);
    prm.q = static_cast<const __half*>(a->q);
    prm.block_tables = a->block_tables;
    prm.context_lens = a->context_lens;
    prm.query_start_loc = a->query_start_loc;
    prm.num_blocks = a->num_blocks;
    prm.num_heads = a->num_heads;
    prm.num_kv_heads = a->num_kv_heads;
    prm.group = a->num_heads / a->num_kv_heads;
    prm.max_blocks_per_seq = a->max_blocks_per_seq;
    prm.max_context_len = a->max_context_len;
    prm.max_query_len = a->max_query_len;
    prm.num_tokens = a->num_tokens;
    prm.scale_log2 = static_cast<float>(static_cast<double>(a->scale) * 1.4426950408889634);
    prm.wait_limit = (o && o->wait_limit) ? o->wait_limit : pa::kDefaultWaitLimit;
    prm.force_timeout = (o && (o->flags & PA_FLAG_FORCE_TIMEOUT)) ? 1 : 0;
    prm.status = pa::device_status_ptr();
    if (!prm.status) return PA_ERR_CUDA;
    prm.trace = g_trace;
    const int tile_tokens = (warp_mma ? 64 : 128) / prm.group;
    dim3 grid((a->max_query_len + tile_tokens - 1) / tile_tokens, a->num_kv_heads, a->num_seqs);
    prm.tiles_per_seq = static_cast<int>(grid.x);
    if (sp.parts) {  // a 1-D grid of units (see PrefixParams::split_parts)
        prm.split_whole = sp.whole;
        prm.split_parts = sp.parts;
        prm.tiles_per_seq = sp.tiles_per_seq;
        prm.split_o = static_cast<float*>(ws);
        prm.split_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + prefix_split_o_bytes(sp, a->head_dim));
        grid = dim3(sp.whole + sp.units * sp.parts, 1, 1);
    }
    if (!warp_mma && !(o && (o->flags & PA_FLAG_PREFIX_GRID))) {
        // the persistent form: the same units, claimed by a grid the SMs hold
        // at once.  Its counter is allocated by the first such call on the
        // stream; a call made while the stream is being captured before that
        // keeps the grid form (allocating would break the capture).
        int num_sms = 0;
        if (query_sm_count(&num_sms) != PA_OK) return PA_ERR_CUDA;
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return PA_ERR_CUDA;
        if (cap == cudaStreamCaptureStatusNone || prefix_sched_ready(stream)) {
            if ((rc = ensure_prefix_sched(stream, &prm.sched))) return rc;
            const long long units = (long long)grid.x * grid.y * grid.z;
            const long long slots = (long long)num_sms * pa::prefix_tc_ctas_per_sm(a->head_dim);
            prm.total_units = static_cast<int>(units);
            grid = dim3(static_cast<unsigned>(units < slots ? units : slots), 1, 1);
        }
    }
    if (o && o->event_partition_begin &&
        cudaEventRecord(static_cast<cudaEvent_t>(o->event_partition_begin), stream) != cudaSuccess)
        return PA_ERR_CUDA;
    const cudaError_t e = warp_mma ? pa::launch_prefix(a->head_dim, prm, maps, grid, stream)
                                   : pa::launch_prefix_tc(a->head_dim, prm, maps, grid, stream);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    if (o && o->event_partition_end &&
        cudaEventRecord(static_cast<cudaEvent_t>(o->event_partition_end), stream) != cudaSuccess)
        return PA_ERR_CUDA;
    if (sp.parts && pa::launch_prefix_merge(a->head_dim, prm, sp.units, stream) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

// Library-owned workspace, one per device, grown on demand.
std::mutex g_ws_mutex;
void* g_ws[kMaxDevices];
size_t g_ws_bytes[kMaxDevices];

int ensure_workspace(size_t need, void** out) {
    *out = nullptr;
    if (need == 0) return PA_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    if (g_ws_bytes[dev] < need) {
        if (g_ws[dev]) {
            // earlier calls may still read the old buffer
            if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
            cudaFree(g_ws[dev]);
            g_ws[dev] = nullptr;
            g_ws_bytes[dev] = 0;
        }
        const size_t grow = align_up(need + need / 4, 1 << 20);
        if (cudaMalloc(&g_ws[dev], grow) != cudaSuccess) {
            cudaGetLastError();
            g_ws[dev] = nullptr;
            return PA_ERR_OOM;
        }
        // the fused combine's tickets must start at zero (every call leaves them so)
        if (cudaMemset(g_ws[dev], 0, grow) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
            cudaFree(g_ws[dev]);
            g_ws[dev] = nullptr;
            return PA_ERR_CUDA;
        }
        g_ws_bytes[dev] = grow;
    }
    *out = g_ws[dev];
    return PA_OK;
}

}  // namespace

extern "C" {

int pa_decode_plan(const pa_decode_args* args, const pa_decode_opts* opts, int num_sms, pa_decode_plan_t* plan) {
    if (!plan || num_sms < 0) return PA_ERR_INVALID_ARG;
    return make_plan(args, opts, num_sms, plan);
}

int pa_decode_ex(const pa_decode_args* args, const pa_decode_opts* opts, void* workspace, size_t workspace_bytes,
                 pa_stream_t stream) {
    pa_decode_plan_t plan;
    int rc = make_plan(args, opts, 0, &plan);
    if (rc) return rc;
    return run(args, opts, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), plan);
}

int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              const int32_t* seq_lens, int num_seqs, int max_blocks_per_seq, int max_seq_len, int64_t num_blocks,
              int num_heads, int num_kv_heads, int head_dim, int block_size, float scale, pa_stream_t stream) {
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
    int rc = make_plan(&a, nullptr, 0, &plan);
    if (rc) return rc;
    void* ws = nullptr;
    rc = ensure_workspace(plan.workspace_bytes, &ws);
    if (rc) return rc;
    return run(&a, nullptr, ws, plan.workspace_bytes, reinterpret_cast<cudaStream_t>(stream), plan);
}

int pa_prefix_ex(const pa_prefix_args* args, const pa_decode_opts* opts, pa_stream_t stream) {
    return run_prefix(args, opts, reinterpret_cast<cudaStream_t>(stream));
}

int pa_prefix_split_workspace_size(const pa_prefix_args* args, const pa_prefix_split_opts* split, size_t* bytes) {
    if (!bytes) return PA_ERR_INVALID_ARG;
    *bytes = 0;
    int rc = validate_prefix(args, nullptr);
    if (rc) return rc;
    int num_sms = 0;
    if (!(split && split->parts) && query_sm_count(&num_sms) != PA_OK) return PA_ERR_CUDA;
    PrefixSplit sp;
    if ((rc = plan_prefix_split(args, split, num_sms, &sp))) return rc;
    *bytes = prefix_split_bytes(sp, args->head_dim);
    return PA_OK;
}

int pa_prefix_split(const pa_prefix_args* args, const pa_decode_opts* opts, const pa_prefix_split_opts* split,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream) {
    return run_prefix(args, opts, reinterpret_cast<cudaStream_t>(stream), true, split, workspace, workspace_bytes);
}

int pa_prefix(void* out, const void* q, const void* k_new, const void* v_new, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* context_lens, const int32_t* query_start_loc, int num_seqs,
              int num_tokens, int max_blocks_per_seq, int max_context_len, int max_query_len, int64_t num_blocks,
              int num_heads, int num_kv_heads, int head_dim, int block_size, float scale, pa_stream_t stream) {
    pa_prefix_args a;
    a.out = out;
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start_loc = query_start_loc;
    a.num_seqs = num_seqs;
    a.num_tokens = num_tokens;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.max_context_len = max_context_len;
    a.max_query_len = max_query_len;
    a.num_blocks = num_blocks;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.scale = scale;
    return run_prefix(&a, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int pa_decode_partials(const pa_decode_args* args, const pa_decode_opts* opts, int partition_size, int partition_begin,
                       int partition_count, float* max_logits, float* exp_sums, float* tmp_out, pa_stream_t stream) {
    return run_partials(args, opts, partition_size, partition_begin, partition_count, max_logits, exp_sums, tmp_out,
                        reinterpret_cast<cudaStream_t>(stream));
}

int pa_merge_partials(void* out, const float* max_logits, const float* exp_sums, const float* tmp_out,
                      const int32_t* seq_lens, int num_seqs, int num_heads, int head_dim, int max_seq_len,
                      int partition_size, int num_sources, int partitions_per_source, pa_stream_t stream) {
    return run_merge(out, max_logits, exp_sums, tmp_out, seq_lens, num_seqs, num_heads, head_dim, max_seq_len,
                     partition_size, num_sources, partitions_per_source, reinterpret_cast<cudaStream_t>(stream));
}

size_t pa_decode_workspace_size(int num_seqs, int max_seq_len, int num_heads, int head_dim, int partition_size) {
    if (num_seqs <= 0 || max_seq_len <= 0 || num_heads <= 0 || head_dim <= 0) return 0;
    if (partition_size > 0)
        return split_workspace_bytes(num_seqs, num_heads, (max_seq_len + partition_size - 1) / partition_size,
                                     head_dim);
    // 0: the most partials an automatic plan makes per (sequence, head):
    // partitions of kDefaultPartition / 2 tokens, or a one-wave plan's (at
    // most 4 CTAs per SM, so at most 4 x SMs partitions, each of at least
    // one block)
    long long parts = (max_seq_len + kDefaultPartition / 2 - 1) / (kDefaultPartition / 2);
    int num_sms = 0;
    if (query_sm_count(&num_sms) != PA_OK || num_sms <= 0) num_sms = kMaxSmsBound;
    const long long one_wave = (max_seq_len + pa::kBlockSize - 1) / pa::kBlockSize;
    parts = std::max(parts, std::min(one_wave, (long long)num_sms * one_wave_ctas_per_sm(head_dim)));
    return split_workspace_bytes(num_seqs, num_heads, static_cast<int>(parts), head_dim);
}

int pa_get_device_status(pa_stream_t stream, int* status) {
    if (!status) return PA_ERR_INVALID_ARG;
    return pa::read_and_clear_status(reinterpret_cast<cudaStream_t>(stream), status) == cudaSuccess ? PA_OK
                                                                                                      : PA_ERR_CUDA;
}

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape (head_dim, block_size or GQA ratio)";
        case PA_ERR_CUDA: return "CUDA runtime error or launch failure";
        case PA_ERR_OOM: return "workspace allocation failed";
        case PA_ERR_WORKSPACE: return "workspace too small or misaligned";
        default: return "unknown status";
    }
}

void pa_release_workspace(void) {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    int cur = 0;
    const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    for (int d = 0; d < kMaxDevices; ++d) {
        if (!g_ws[d]) continue;
        if (cudaSetDevice(d) == cudaSuccess) {
            cudaDeviceSynchronize();
            cudaFree(g_ws[d]);
        }
        g_ws[d] = nullptr;
        g_ws_bytes[d] = 0;
    }
    std::lock_guard<std::mutex> lock_sched(g_sched_mutex);
    for (const auto& e : g_sched) {
        if (cudaSetDevice(e.first.first) == cudaSuccess) {
            cudaDeviceSynchronize();
            cudaFree(e.second);
        }
    }
    g_sched.clear();
    if (have_cur) cudaSetDevice(cur);
}

int pa_version(void) { return 100; }

#ifdef PA_TRACE
// Diagnostic builds only (not part of the public header).
void pa_debug_set_trace(void* device_buffer) { g_trace = static_cast<unsigned long long*>(device_buffer); }
#endif

}  // extern "C"
