// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05),
// one CTA pair (two SMs) per work item.
//
// Same operation as the mma.sync kernel in prefill.cu: query j of a chunk of n
// tokens of a sequence with L cached tokens attends causally to tokens
// 0 .. L-n+j (caffein.top, "Chunked Prefill"), K/V gathered through the block
// table.  Used for bf16 caches with head_dim 128.
//
// Work item: (sequence, tile of 256 packed query rows, kv head); row R of the
// tile is query position R / G, head kvh*G + R % G, so the G heads of a kv
// head share every K/V tile.  A cluster of two CTAs takes each item: the even
// CTA holds rows 0-127, the odd CTA rows 128-255, and threads of the even CTA
// issue every MMA in the pair form (tcgen05 cta_group::2, M = 256), which
// runs on both SMs' tensor cores at once:
//   S(g)  = Q K(g)^T : M=256, N=128 keys, K=d; A = Q (each CTA its 128 rows),
//                      B = K (each CTA 64 of the 128 keys), S in each CTA's
//                      tensor memory (its 128 rows x 128 keys);
//   O    += P(g) V(g): M=256, N=d, K=128 keys; A = P from each CTA's tensor
//                      memory, B = V (each CTA 64 of the 128 columns of d).
// One MMA instruction does both SMs' work, and each SM loads only half of
// every K and V tile.  (Measured on GB300: one thread issues a tcgen05.mma
// about every 64 cycles whatever its N, and one thread issues a 2 KB TMA box
// about every 130-180 cycles.)
//
// The key tiles of an item run through double buffers: S of tile g in one of
// two tensor-memory buffers, its P in one of two others, so that S(g+2) is
// computed while the softmax still works on S(g), and PV(g) while it works on
// S(g+1).  The tensor pipe then runs without waiting for the softmax, which
// is the bound when each S buffer has to hold its P until PV has read it.
// Warp roles (one CTA per SM, 14 warps, in both CTAs of the pair):
//   * 8 softmax warps.  Warp w owns rows 32 (w % 4) .. +31 of its CTA (its
//     tensor-memory lanes) and keys 64 (w / 4) .. +63 of every tile, so two
//     threads share each row.  A thread reads its 64 scores in one load,
//     whose own reduction gives their maximum, releases the S buffer, masks,
//     trades maxima with the other thread of its row through shared memory,
//     computes p = 2^(s * scale * log2 e - m) (one paired multiply-add per
//     two elements, ex2.approx on the special-function unit) and stores its
//     64 keys of P as bf16 pairs; P(g) goes to the PV lane once all 8 warps
//     of both CTAs have stored it (either half's PV writes the whole O row,
//     which both threads of the row may have to rescale first).  Both
//     threads of a row keep the same reference max m, one O row and a
//     partial row sum, added at the end.
//   * two MMA-issuing lanes in the even CTA: lane 0 of warp 8 issues every
//     S(g) (once K(g) has landed and S(g-2) has been read out of the
//     buffer), lane 0 of warp 9 every PV(g) (once V(g) has landed and P(g)
//     is stored).  They write disjoint tensor
//     memory and need no order between them.
//   * four loader warps per CTA, two for K and two for V, that gather this
//     CTA's half of each tile through the block table with 2-D TMA boxes (the
//     cache viewed as [num_blocks * num_kv_heads * 16 rows][128] with 128-byte
//     swizzle, which writes exactly the layout the MMAs read), reading the
//     table one tile ahead.  K: this CTA's 4 blocks of the tile's 8 (2 per
//     warp), both 64-column halves; blocks past the keys are not loaded
//     (their scores are masked).  V: all 8 blocks (4 per warp), this CTA's
//     64 columns; rows past the keys are zeroed in place (P = 0 times a NaN
//     in an unused row would still poison O) and a block that the keys end
//     inside is copied with zero-filling cp.async.  Every load of either CTA
//     counts its bytes on the even CTA's barrier of that stage, where the
//     MMA lane waits; a stage is refilled when the S (for K) or PV (for V)
//     that read it has finished.  The first K loader also loads this CTA's
//     Q rows of each item (TMA, 3-D box) and, in the even CTA, hands out the
//     items.
// The running max of a row is only moved when a tile maximum exceeds it by
// more than 8 (log2 units), so P <= 256 and O is rarely rescaled; numerator
// and denominator share the same reference, so the result is exact.
//
// TMEM columns (all 512, in each CTA): S of tile g at 128 (g % 2), O at 256,
// P of tile g at 384 + 64 (g % 2).  Shared memory per CTA, in the
// 128-byte-swizzled canonical layout (8-row atoms of 8 x 128 bytes, 16-byte
// chunk c of row r at chunk c ^ (r % 8)):
//   Q : two 64-column halves of this CTA's 128 rows              (32 KB)
//   K : six stages x two 64-column halves of this CTA's 64 keys  (96 KB)
//   V : four stages x 128 keys of this CTA's 64 columns          (64 KB)
// Waits.  Every wait on an mbarrier is bounded in time (PrefillParams::
// wait_ns, from %globaltimer); the two warps that share rows meet at a named
// barrier once per tile, and a warp that leaves after a failure releases its
// partner from it.  A wait that
// runs out makes the whole warp leave its role loop (the decision is taken
// warp-wide, so no lane is left at a warp barrier) and raises an abort flag
// in both CTAs, at which the other roles' waits give up too.  A role that
// has left issues no further copies or MMAs.  At the end one thread of each
// CTA waits for both MMA lanes' final commits, which arrive after every
// earlier one (a separate, fixed bound of one second), the pair meets at a
// cluster barrier, and if anything failed (every failure raises the abort
// flag in both CTAs, so both take the same branch) both CTAs wait 100 us
// more, so that copies already issued land before either CTA's shared
// memory is released, and meet again; the CTA records PKV_STATUS_INTERNAL,
// frees its tensor memory and returns.
// (A failure stops all further issue, so the only copies that can still be
// in flight were issued before it; a TMA load or cp.async of a few KB lands
// within microseconds.  Waiting on their barriers instead is not possible:
// after a failure a phase may never collect all its arrivals.)
#include <math.h>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>
#include <mutex>
#include <string.h>

#include "common.cuh"
#include "prefill_common.cuh"
#include "tcgen05.cuh"

namespace {

using pkv::kBlock;
using pkv::PrefillParams;
namespace tc = pkv::tc;

constexpr int D = 128;
constexpr int BM = 128;         // query rows per CTA
constexpr int kPairRows = 256;  // query rows per work item (both CTAs)
constexpr int BN = 128;         // keys per tile
constexpr int kSoftmaxThreads = 256;  // warps 0-7
constexpr int kSWarp = 8, kPVWarp = 9;  // the even CTA's MMA lanes: S = Q K^T, and O += P V
constexpr int kLoadWarp0 = 10;          // 10, 11: K loaders; 12, 13: V loaders
constexpr int kThreads = 14 * 32;
constexpr uint32_t kTmemCols = 512;
// S of tile g in columns 128 (g % 2); O at 256; P of tile g at 384 + 64 (g % 2)
constexpr uint32_t kOCol = 256, kPCol = 384;
constexpr int kKStages = 6, kVStages = 4;

constexpr int kQHalf = BM * 128;        // 16 KB: 128 rows x 64 bf16
constexpr int kQBytes = 2 * kQHalf;     // 32 KB
constexpr int kKHalf = 64 * 128;        // 8 KB: this CTA's 64 keys x 64 bf16
constexpr int kKStage = 2 * kKHalf;     // 16 KB
constexpr int kVStage = BN * 128;       // 16 KB: 128 keys x this CTA's 64 bf16
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;                  // 32768
constexpr int kOffV = kOffK + kKStages * kKStage;       // 131072
constexpr int kOffBar = kOffV + kVStages * kVStage;     // 196608

// mbarrier indices.  "both": each CTA has its own, signalled for both by the
// even CTA's MMA commits.  "even": used in the even CTA only, which both
// CTAs' threads (or copies) arrive at.
enum Bar : int {
    B_PFULL = 0,   // [g % 2][half] P(g) of keys 64h .. 64h+63 stored; even, its 4 warps per CTA
    B_SFREE = 4,   // [g % 2] S(g) read into registers by every softmax warp; even, 8 warps per CTA
    B_KFULL = 6,   // [stage] K tile landed; even, 2 loaders per CTA + bytes
    // [stage] the S reading the stage is done; both.  Also the softmax
    // warps' "S(g) computed": its next phase needs S(g + 6), which the
    // warps' own reads of S(g + 4) hold back
    B_KEMPTY = B_KFULL + kKStages,
    B_VFULL = B_KEMPTY + kKStages,   // [stage] V tile landed; even, 2 loaders per CTA + bytes
    // [stage] the PV reading the stage is done; both.  Also the softmax
    // warps' "PV(g) done": P(g) buffer free, O holds every tile up to g
    B_VEMPTY = B_VFULL + kVStages,
    B_GO = B_VEMPTY + kVStages,      // [k & 1] Q of the k-th item with work landed; even
    B_ITEM_FULL = B_GO + 2,          // [slot] item published; both
    B_ITEM_EMPTY = B_ITEM_FULL + 2,  // [slot] every reader of both CTAs has read it; even
    B_DONE = B_ITEM_EMPTY + 2,       // all MMAs finished (each lane's last commit); both
    B_QFREE = B_DONE + 1,            // every S of the k-th item with work finished; both
    B_EPI = B_QFREE + 1,             // the k-th item's O read by both CTAs' softmax warps; even, 16 warps
    kNumBars = B_EPI + 1,
};
// item queue readers: even CTA: K loader 1, V loaders, two MMA lanes and 8
// softmax warps; odd CTA: four loaders and 8 softmax warps
constexpr int kItemReaders = 25;
constexpr int kOffSlots = (kOffBar + kNumBars * 8 + 15) & ~15;  // TMEM address (16 B), two item slots, abort flag
static_assert(kOffSlots % 16 == 0, "item slots are 16-byte vectors");
constexpr int kOffAbort = kOffSlots + 16 + 2 * 16;
// Row exchange between the two threads that share a row: [slot][half][row]
// floats; slots 0 and 1 carry tile maxima (by tile parity), 2 and 3 row sums
// (by item parity).
constexpr int kOffX = kOffAbort + 16;
constexpr int kXBytes = 4 * 2 * BM * 4;
constexpr int kSmemBytes = kOffX + kXBytes;
static_assert(kOffX % 4 == 0, "exchange words are 4-byte aligned");
static_assert(kSmemBytes <= 232448, "more shared memory than a CTA may have");
static_assert(kSmemBytes > 232448 / 2, "one CTA per SM: the tensor memory is all allocated by one CTA");

constexpr unsigned long long kDrainNs = 1000000000ull;  // the final wait for this CTA pair's MMAs
constexpr unsigned long long kGraceNs = 100000ull;      // after a failure, for copies in flight
constexpr unsigned long long kDefaultWaitNs = 200000000ull;

// S: M = 256 rows over the pair, N = 128 keys, both operands K-major.
constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kPairRows, BN, false, false);
// PV: M = 256, N = d = 128, B = V is MN-major (d contiguous).
constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(kPairRows, D, false, true);

__device__ __forceinline__ int sw128(int r, int c16) {
    return (r >> 3) * 1024 + (r & 7) * 128 + ((c16 ^ (r & 7)) << 4);
}

// The next work item for this cluster: items below the number of clusters
// are each cluster's first; later ones are handed out in order by a counter
// in the workspace.  The counter is the pair {launch tag, count} (16 bytes):
// the first fetch of a launch finds another tag (an earlier launch's, or
// whatever the workspace held) and installs {its tag, 0} with one 16-byte
// compare-and-swap, so the call needs no clearing pass before the kernel.
// Tags are 64-bit values drawn per launch; only a launch's own tag can match.
__device__ __forceinline__ int next_item(const PrefillParams &p) {
    const unsigned long long k = pkv::tagged_add(p.item_counter, p.launch_tag);
    const unsigned long long item = (unsigned long long)(gridDim.x / 2) + k;
    return item < (unsigned long long)p.num_items ? (int)item : 0x7fffffff;
}

// Count this CTA in the second pair of the workspace counter, {launch tag,
// CTAs done}, installed like the first: the even CTA once its queue has made
// its last fetch, the odd CTA (which fetches nothing) at once.  The launch's
// last count clears both tags, so the next launch installs its own pairs
// even when it carries this launch's tag: a launch replayed from a CUDA
// graph keeps the parameters, tag included, that it was captured with.  (By
// then every CTA has made its last fetch from the first pair.)
__device__ __forceinline__ void count_exit(const PrefillParams &p) {
    const unsigned long long k = pkv::tagged_add(p.item_counter + 2, p.launch_tag);
    if (k == (unsigned long long)gridDim.x - 1) {
        atomicExch(p.item_counter, 0ull);
        atomicExch(p.item_counter + 2, 0ull);
    }
}

// The queue's record of item `item`: (item, first query, queries, length).
__device__ __forceinline__ int4 item_record(const PrefillParams &p, int item) {
    int4 v = make_int4(item, 0, 0, 0);
    if (item < p.num_items && p.prefix_len) {
        v.y = 0;  // the decode queries, one "position" per sequence
        v.z = p.max_q_len;
        v.w = p.prefix_len;
    } else if (item < p.num_items) {
        const int s = p.num_seqs - 1 - item / (p.num_kv_heads * p.tiles_per_seq);
        v.y = p.cu_q_lens[s];
        v.z = p.cu_q_lens[s + 1] - v.y;
        v.w = p.context_lens[s];
    }
    return v;
}

// Item (sequence, pair tile, kv head) as published in the shared-memory
// queue: (item, q0, n, L); every role of both CTAs derives the rest.
struct ItemInfo {
    int item, s, kvh, tile, q0, n, L, nkt, kv_end, mask_from, row0;
    bool stop, skip, bad_len, bad_qlen;
};

__device__ __forceinline__ ItemInfo item_info(const PrefillParams &p, int4 v, uint32_t rank) {
    ItemInfo it;
    it.item = v.x;
    it.q0 = v.y;
    it.n = v.z;
    it.L = v.w;
    it.stop = v.x >= p.num_items;
    // later sequences first, later q tiles (more keys) first within a sequence
    const int per_seq = p.num_kv_heads * p.tiles_per_seq;
    const int zi = it.stop ? 0 : v.x / per_seq;
    const int rem = it.stop ? 0 : v.x - zi * per_seq;
    it.s = p.num_seqs - 1 - zi;
    it.tile = p.tiles_per_seq - 1 - rem / p.num_kv_heads;
    it.kvh = rem - (rem / p.num_kv_heads) * p.num_kv_heads;
    it.row0 = it.tile * kPairRows + (int)rank * BM;  // this CTA's first packed row
    it.bad_len = !it.stop && (it.L < 0 || it.L > p.len_cap);
    it.bad_qlen = !it.stop && !it.bad_len && !p.prefix_len &&
                  (it.q0 < 0 || it.n < 0 || it.n > it.L || it.n > p.max_q_len || it.q0 + it.n > p.total_q);
    it.skip = it.stop || it.bad_len || it.bad_qlen || it.tile * kPairRows >= it.n * p.group;
    if (it.skip) {
        it.nkt = it.kv_end = it.mask_from = 0;
    } else if (p.prefix_len) {  // every query sees the whole shared prefix, nothing after it
        it.kv_end = it.mask_from = p.prefix_len;
        it.nkt = (p.prefix_len + BN - 1) / BN;
    } else {
        // both CTAs walk the key tiles of the pair's last row
        const int prior = it.L - it.n;
        const int j_last = min(it.n - 1, (it.tile * kPairRows + kPairRows - 1) / p.group);
        it.kv_end = prior + j_last + 1;
        it.nkt = (it.kv_end + BN - 1) / BN;
        it.mask_from = prior + it.row0 / p.group + 1;  // keys below this need no causal mask in this CTA
    }
    return it;
}

template <typename OutT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_q,
                      const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v) {
    extern __shared__ __align__(1024) unsigned char smem[];
    // a dependent launch (the decode partitions beside the shared-prefix
    // mode) may start as soon as every CTA of this one has
    pkv::allow_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.group;
    const uint32_t rank = tc::cluster_rank();
    const bool even = rank == 0;
    const uint32_t sbase = pkv::smem_u32(smem);
    // The same dynamic shared-memory base in both CTAs: one alignment
    // decision for the pair.
    const bool misaligned = (sbase & 1023u) != 0;

    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffSlots);
    int4 *item_slots = reinterpret_cast<int4 *>(smem + kOffSlots + 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffAbort);
    float *xch = reinterpret_cast<float *>(smem + kOffX);
    // shared::cta address of barrier i, and the shared::cluster windows of
    // the even CTA, this CTA and the other CTA
    auto bar = [&](int i) { return sbase + kOffBar + 8u * (uint32_t)i; };
    const uint32_t base_even = tc::mapa(sbase, 0), base_own = tc::mapa(sbase, rank),
                   base_other = tc::mapa(sbase, rank ^ 1u);
    auto bar_even = [&](int i) { return base_even + kOffBar + 8u * (uint32_t)i; };
    auto bar_own = [&](int i) { return base_own + kOffBar + 8u * (uint32_t)i; };
    auto bar_other = [&](int i) { return base_other + kOffBar + 8u * (uint32_t)i; };

    // While the barriers and tensor memory are set up: the tensor maps into
    // the TMA unit's cache, the first item's block-table row into L2, and
    // (queue warp) the first item's record into registers.
    int4 first_rec = make_int4(0, 0, 0, 0);
    if (warp >= kLoadWarp0 && lane == 0 && !misaligned) {
        const int item = (int)(blockIdx.x >> 1);
        if (warp == kLoadWarp0) {
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_k)) : "memory");
            if (p.q_tma) asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_q)) : "memory");
            if (even) first_rec = item_record(p, item);
        } else if (warp == kLoadWarp0 + 2) {
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_v)) : "memory");
        }
        if (item < p.num_items) {
            const int s = p.prefix_len ? 0 : p.num_seqs - 1 - item / (p.num_kv_heads * p.tiles_per_seq);
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p.block_tables + (size_t)s * p.max_blocks) : "memory");
        }
    }
    if (tid == 0 && !misaligned) {
        uint64_t *b = reinterpret_cast<uint64_t *>(smem + kOffBar);
        for (int t = 0; t < 2; t++) {
            tc::mbar_init(b + B_PFULL + 2 * t, 8);
            tc::mbar_init(b + B_PFULL + 2 * t + 1, 8);
            tc::mbar_init(b + B_SFREE + t, 16);
            tc::mbar_init(b + B_ITEM_FULL + t, 1);
            tc::mbar_init(b + B_ITEM_EMPTY + t, kItemReaders);
            // Q lands by TMA (each CTA's first K loader arrives with its
            // bytes) or by the softmax threads' copies (8 warps in each CTA)
            tc::mbar_init(b + B_GO + t, p.q_tma ? 2 : 16);
        }
        tc::mbar_init(b + B_DONE, 2);  // one final commit per issuing lane
        tc::mbar_init(b + B_QFREE, 1);
        tc::mbar_init(b + B_EPI, 16);
        for (int st = 0; st < kKStages; st++) {
            tc::mbar_init(b + B_KFULL + st, 4);
            tc::mbar_init(b + B_KEMPTY + st, 1);
        }
        for (int st = 0; st < kVStages; st++) {
            tc::mbar_init(b + B_VFULL + st, 4);
            tc::mbar_init(b + B_VEMPTY + st, 1);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0 && !misaligned) {
        tc::tmem_alloc_pair(tmem_slot, kTmemCols);
        tc::tmem_relinquish_pair();
    }
    tc::fence_before_sync();
    tc::cluster_sync();  // both CTAs' barriers initialised and tensor memory allocated
    tc::fence_after_sync();
    const uint32_t tmem = misaligned ? 0u : *tmem_slot;

    bool failed = misaligned;
    // Give up on every other wait of both CTAs (after a wait ran out).
    auto raise_abort = [&]() {
        *abort_flag = 1;
        asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(base_other + kOffAbort), "r"(1) : "memory");
    };
    // Bounded wait for phase `parity` of this CTA's barrier i by the calling
    // thread; false when the time budget ran out or another role aborted.
    // The item queue's hand-offs carry shared-memory data across the pair
    // and are acquired at cluster scope; the others at the default (CTA)
    // scope, whose data (tensor memory, copies counted in bytes) is ordered
    // by other means: a cluster-scope release / acquire on every tile costs
    // microseconds per item.
    auto wait1 = [&](int i, unsigned parity) -> bool {
        const uint32_t a = bar(i);
        const bool cl = i >= B_ITEM_FULL && i < B_DONE;
        if (cl ? tc::mbar_test_cluster(a, parity) : tc::mbar_test_cta(a, parity)) return true;
        const unsigned long long t0 = tc::globaltimer_ns();
        for (;;) {
            if (cl ? tc::mbar_try_cluster(a, parity) : tc::mbar_try_cta(a, parity)) return true;
            if (*abort_flag) return false;
            if (tc::globaltimer_ns() - t0 > p.wait_ns) return false;
        }
    };
    // The same waited by every lane of the warp, with one warp-wide outcome.
    auto wait_warp = [&](int i, unsigned parity) -> bool {
        const bool ok = __all_sync(0xffffffffu, wait1(i, parity));
        if (!ok) {
            failed = true;
            if (lane == 0) raise_abort();
        }
        return ok;
    };
    // Waited by lane 0 only, outcome broadcast to the warp.
    auto wait_lane0 = [&](int i, unsigned parity) -> bool {
        int ok = 1;
        if (lane == 0) ok = wait1(i, parity) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            failed = true;
            if (lane == 0) raise_abort();
        }
        return ok != 0;
    };
    // Take item i from this CTA's queue (every role reads every item): lane 0
    // waits, the warp reads, lane 0 reports the slot read to the even CTA.
    // The stop record is the last one: no slot is refilled after it, so it is
    // not reported read (the cluster-scope release of that report would wait
    // for the reader's output stores to complete).
    auto take_item = [&](int i, ItemInfo &it) -> bool {
        if (!wait_lane0(B_ITEM_FULL + (i & 1), (unsigned)((i >> 1) & 1))) return false;
        const int4 v = item_slots[i & 1];
        __syncwarp();
        it = item_info(p, v, rank);
        if (lane == 0 && !it.stop) tc::mbar_arrive_cluster(bar_even(B_ITEM_EMPTY + (i & 1)));
        return true;
    };

    // Running counts that carry the barrier phases from one item to the next:
    // key tiles of the items with work so far (the global tile index g of
    // an item's tile t is g0 + t: S, P and ring buffers and their phases) and
    // items with work (the Q, epilogue and exchange phases).  Every role of
    // both CTAs walks the same items, so every role's counts agree.
    int g0 = 0, go_count = 0;
    auto advance = [&](const ItemInfo &it) {
        g0 += it.nkt;
        go_count += it.skip ? 0 : 1;
    };

    if (failed) {
        // nothing but the exit count: misaligned shared memory (reported below)
        if (tid == 0) count_exit(p);
    } else if (warp >= kLoadWarp0) {
        // ---------------- loaders: two for K (each 2 of this CTA's 4 blocks
        // of a tile, both 64-column halves) and two for V (each 4 of the 8
        // blocks, this CTA's 64 columns); a thread issues a TMA box only
        // every 130-180 cycles, so each tile's 16 boxes are split over four
        // warps.  The even CTA's first K loader also runs the item queue,
        // and each CTA's first K loader loads its Q rows.
        const int lw = warp - kLoadWarp0;
        const bool is_k = lw < 2;
        const int sub = lw & 1;
        const bool runs_queue = is_k && sub == 0 && even;
        const int full0 = is_k ? B_KFULL : B_VFULL, empty0 = is_k ? B_KEMPTY : B_VEMPTY;
        const int nstage = is_k ? kKStages : kVStages;
        const unsigned char *cache = static_cast<const unsigned char *>(is_k ? p.k_cache : p.v_cache);
        int item = (int)(blockIdx.x >> 1);  // the cluster's first item; later ones come from the counter
        for (int i = 0;; i++) {
            ItemInfo it;
            if (runs_queue) {
                int4 v = make_int4(item, 0, 0, 0);
                if (i >= 2 && !wait_lane0(B_ITEM_EMPTY + (i & 1), (unsigned)(((i >> 1) - 1) & 1))) break;
                if (lane == 0) {
                    v = i == 0 ? first_rec : item_record(p, item);
                    item_slots[i & 1] = v;
                    tc::st_cluster_v4(base_other + kOffSlots + 16 + 16 * (i & 1), v);
                    // release: each slot is visible to its CTA's waiters
                    tc::mbar_arrive_cluster(bar_own(B_ITEM_FULL + (i & 1)));
                    tc::mbar_arrive_cluster(bar_other(B_ITEM_FULL + (i & 1)));
                }
                v.x = __shfl_sync(0xffffffffu, v.x, 0);
                v.y = __shfl_sync(0xffffffffu, v.y, 0);
                v.z = __shfl_sync(0xffffffffu, v.z, 0);
                v.w = __shfl_sync(0xffffffffu, v.w, 0);
                it = item_info(p, v, rank);
                if (lane == 0 && it.tile == 0 && it.kvh == 0) {
                    if (it.bad_len) pkv::flag(p.status, PKV_STATUS_BAD_LENGTH);
                    if (it.bad_qlen) pkv::flag(p.status, PKV_STATUS_BAD_QLEN);
                }
            } else if (!take_item(i, it)) {
                break;
            }
            if (it.stop) break;
            if (is_k && sub == 0 && p.q_tma && !it.skip) {
                // This CTA's q rows, as soon as the previous item's S MMAs are
                // done with the buffer: they land while that item finishes.
                // Row r = j * G + h is query q0 + row0/G + j, head kvh*G + h:
                // one 3-D box {64 columns, G heads, 128/G queries} per half.
                // Rows past the chunk read other queries or zeros and are
                // masked.
                if (go_count > 0 && !wait_warp(B_QFREE, (unsigned)((go_count - 1) & 1))) break;
                if (lane == 0) {
                    const uint32_t go = bar_even(B_GO + (go_count & 1));
                    tc::mbar_arrive_expect_tx_remote(go, kQBytes);
                    const int z = it.q0 + it.row0 / G;
#pragma unroll
                    for (int h = 0; h < 2; h++)
                        tc::tma_load_3d_pair(smem + kOffQ + h * kQHalf, &tmap_q, h * 64, it.kvh * G, z, go);
                }
            }
            const int32_t *table = p.block_tables + (size_t)(it.skip ? 0 : it.s) * p.max_blocks;
            const int nb = is_k ? 2 : 4;                                   // blocks of a tile this warp loads
            const int b0 = is_k ? 4 * (int)rank + 2 * sub : 4 * sub;       // the first of them
            // Block ids of this warp's blocks of tile t (lane q < nb: block
            // b0 + q), -1 past the keys.  They are read one tile ahead, so the
            // copies of a tile never wait for its table entries.
            auto table_id = [&](int t) {
                int id = -1;
                if (t < it.nkt && lane < nb && t * BN + (b0 + lane) * kBlock < it.kv_end) id = table[t * 8 + b0 + lane];
                return id;
            };
            int next_id = table_id(0);
            bool ok = true;
            for (int t = 0; t < it.nkt; t++) {
                const int g = g0 + t, st = g % nstage;
                // the stage's previous tile (g - nstage) has been read
                if (g >= nstage && !(ok = wait_warp(empty0 + st, (unsigned)((g / nstage - 1) & 1)))) break;
                const int my_id = next_id;
                next_id = table_id(t + 1);
                const uint32_t full = bar_even(full0 + st);
                const int tile_keys = min(BN, it.kv_end - t * BN);
                const int nbk = (tile_keys + kBlock - 1) / kBlock;  // blocks of the tile holding keys
                const int box_rows = p.num_blocks * p.num_kv_heads * kBlock;  // rows of the 2-D view
                if (is_k) {
                    // this warp's blocks holding keys (the rest are masked out of S)
                    unsigned char *dst = smem + kOffK + st * kKStage;
                    const int nk = max(0, min(2, nbk - b0));
                    int y = box_rows;
                    if (lane < nk) {
                        if (my_id >= 0 && my_id < p.num_blocks)
                            y = (my_id * p.num_kv_heads + it.kvh) * kBlock;
                        else
                            pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                    }
                    const int y0 = __shfl_sync(0xffffffffu, y, 0), y1 = __shfl_sync(0xffffffffu, y, 1);
                    if (lane == 0) {
                        tc::mbar_arrive_expect_tx_remote(full, (uint32_t)(nk * 2 * 2048));
                        // block b0 + q is this CTA's block 2 sub + q of the tile
#pragma unroll
                        for (int q = 0; q < 2; q++) {
                            if (q >= nk) break;
#pragma unroll
                            for (int h = 0; h < 2; h++)
                                tc::tma_load_2d_pair(dst + h * kKHalf + (2 * sub + q) * 2048, &tmap_k,
                                                     h * 64, q ? y1 : y0, full);
                        }
                    }
                } else {
                    // blocks b0 .. b0+3, this CTA's 64 columns of d; a block
                    // that the keys end inside by zero-filling copies, rows
                    // past the keys zeroed
                    unsigned char *dst = smem + kOffV + st * kVStage;
                    const int cpq = (tile_keys % kBlock) ? tile_keys / kBlock : -1;
                    const int ntma = cpq >= 0 ? nbk - 1 : nbk;  // blocks 0 .. ntma-1 of the tile by TMA
                    const int my_ntma = max(0, min(4, ntma - b0));
                    int y = box_rows;
                    if (lane < my_ntma) {
                        if (my_id >= 0 && my_id < p.num_blocks)
                            y = (my_id * p.num_kv_heads + it.kvh) * kBlock;
                        else
                            pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                    }
                    int ys[4];
#pragma unroll
                    for (int q = 0; q < 4; q++) ys[q] = __shfl_sync(0xffffffffu, y, q);
                    const int r_lo = max(kBlock * ntma, kBlock * b0), r_hi = kBlock * (b0 + 4);
                    if (r_lo < r_hi) {
                        // generic-proxy part of this warp's rows: the partial
                        // block's live rows by zero-filling copies, every
                        // other row past the keys zeroed with stores
                        const bool mine = cpq >= b0 && cpq < b0 + 4;
                        const int phys = mine ? __shfl_sync(0xffffffffu, my_id, cpq - b0) : 0;
                        const bool bok = phys >= 0 && phys < p.num_blocks;
                        if (mine && !bok && lane == 0) pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                        for (int e = lane + 8 * r_lo; e < 8 * r_hi; e += 32) {
                            const int r = e >> 3, c = e & 7;
                            unsigned char *d = dst + sw128(r, c);
                            if (r < tile_keys) {
                                const int rb = r % kBlock;
                                const size_t go =
                                    bok ? ((((size_t)phys * p.num_kv_heads + it.kvh) * kBlock + rb) * D + rank * 64) * 2 +
                                              c * 16
                                        : 0;
                                pkv::cp_async16(d, cache + go, bok ? 16 : 0);
                            } else {
                                *reinterpret_cast<uint4 *>(d) = make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                        pkv::cp_async_commit();
                        pkv::cp_async_wait<0>();
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                    }
                    if (lane == 0) {
                        tc::mbar_arrive_expect_tx_remote(full, (uint32_t)(my_ntma * 2048));
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            if (q >= my_ntma) break;
                            tc::tma_load_2d_pair(dst + (b0 + q) * 2048, &tmap_v, (int)rank * 64, ys[q], full);
                        }
                    }
                }
            }
            if (!ok) break;
            advance(it);
            if (runs_queue) {  // the next item, fetched while the consumers work on this one
                if (lane == 0) item = next_item(p);
                item = __shfl_sync(0xffffffffu, item, 0);
            }
        }
        // this CTA's fetches are over (the odd CTA makes none)
        if (runs_queue && lane == 0) count_exit(p);
    } else if (warp == kSWarp || warp == kPVWarp) {
        // ---------------- MMA issue: lane 0 of warp 8 of the even CTA issues
        // every S = Q K^T of the pair, lane 0 of warp 9 every O += P V.  The
        // two lanes write disjoint tensor memory (the two S buffers; O), so
        // neither orders itself after the other: S(g+2) goes out as soon as
        // the softmax warps have read S(g) into registers, while they still
        // work on it, and PV(g) as soon as they have stored P(g).
        if (!even && warp == kPVWarp && lane == 0) count_exit(p);  // the odd CTA fetches no item
        if (even && lane == 0) {
            // one commit per CTA of the pair: each CTA's barrier i
            auto commit_both = [&](int i) {
                tc::mma_commit_pair(bar_own(i));
                tc::mma_commit_pair(bar_other(i));
            };
            if (warp == kSWarp) {
                // Descriptors of the first 16 columns of Q and of stage 0 of
                // the K ring; a stage, a half or 16 more columns is a constant
                // number of 16-byte units on.
                const uint64_t q_desc = tc::smem_desc_sw128(sbase + kOffQ, 16, 1024);
                const uint64_t k_desc0 = tc::smem_desc_sw128(sbase + kOffK, 16, 1024);
                for (int i = 0;; i++) {
                    // Take item i alone (the other lanes idle).  The slot is
                    // reported read only after this item's Q barrier has been
                    // waited for: the queue then cannot run two items ahead
                    // of this lane, so neither Q barrier can complete a phase
                    // that this lane has not yet waited for.
                    if (!wait1(B_ITEM_FULL + (i & 1), (unsigned)((i >> 1) & 1))) { failed = true; break; }
                    const ItemInfo it = item_info(p, item_slots[i & 1], rank);
                    if (!it.stop && !it.skip && !wait1(B_GO + (go_count & 1), (unsigned)((go_count >> 1) & 1))) {
                        failed = true;
                        break;
                    }
                    if (it.stop) break;
                    tc::mbar_arrive_cluster(bar_own(B_ITEM_EMPTY + (i & 1)));
                    for (int t = 0; t < it.nkt && !failed; t++) {
                        const int g = g0 + t, st = g % kKStages;
                        // the softmax warps have read S(g-2) out of this buffer
                        if (g >= 2 && !wait1(B_SFREE + (g & 1), (unsigned)(((g - 2) >> 1) & 1))) { failed = true; break; }
                        if (!wait1(B_KFULL + st, (unsigned)((g / kKStages) & 1))) { failed = true; break; }
                        tc::fence_after_sync();
                        tc::mma_s_tile_pair<kQHalf / 16, kKHalf / 16>(tmem + (uint32_t)((g & 1) * BN), q_desc,
                                                                       k_desc0 + (uint64_t)(st * (kKStage / 16)), kIdescS);
                        commit_both(B_KEMPTY + st);
                        if (t + 1 == it.nkt) commit_both(B_QFREE);  // the item's last read of Q
                    }
                    if (failed) break;
                    advance(it);
                }
            } else {
                // V is MN-major: the next 8 keys at +1 KB (SBO); this CTA's
                // 64 columns are one 128-byte swizzle span (LBO unused).
                const uint64_t v_desc0 = tc::smem_desc_sw128(sbase + kOffV, kVStage, 1024);
                for (int i = 0;; i++) {
                    if (!wait1(B_ITEM_FULL + (i & 1), (unsigned)((i >> 1) & 1))) { failed = true; break; }
                    const ItemInfo it = item_info(p, item_slots[i & 1], rank);
                    if (it.stop) break;
                    tc::mbar_arrive_cluster(bar_own(B_ITEM_EMPTY + (i & 1)));
                    if (it.skip) {
                        advance(it);
                        continue;
                    }
                    // The previous item's O has been read by both CTAs before
                    // this item's first PV overwrites it.
                    if (go_count > 0 && !wait1(B_EPI, (unsigned)((go_count - 1) & 1))) { failed = true; break; }
                    for (int t = 0; t < it.nkt && !failed; t++) {
                        const int g = g0 + t, st = g % kVStages;
                        if (!wait1(B_VFULL + st, (unsigned)((g / kVStages) & 1))) { failed = true; break; }
                        // both halves of P(g) stored in both CTAs: either half's
                        // PV writes every column of O, which the softmax threads
                        // of both halves may rescale before they store P(g)
                        if (!wait1(B_PFULL + 2 * (g & 1), (unsigned)((g >> 1) & 1)) ||
                            !wait1(B_PFULL + 2 * (g & 1) + 1, (unsigned)((g >> 1) & 1))) {
                            failed = true;
                            break;
                        }
                        tc::fence_after_sync();
                        for (int h = 0; h < 2; h++) {
                            tc::mma_pv_half_pair<2048 / 16>(
                                tmem + kOCol, tmem + kPCol + (uint32_t)((g & 1) * 64 + h * 32),
                                v_desc0 + (uint64_t)(st * (kVStage / 16) + h * 4 * (2048 / 16)), kIdescPV,
                                (t == 0 && h == 0) ? 0u : 1u);
                        }
                        commit_both(B_VEMPTY + st);
                    }
                    if (failed) break;
                    advance(it);
                }
            }
            if (failed) raise_abort();
            // every MMA of this lane has finished, and every earlier commit
            // of it has arrived at this CTA's barriers, before the tensor
            // memory is released
            commit_both(B_DONE);
        }
        if (warp == kSWarp && lane == 0) {
            // in both CTAs: both lanes' final commits have arrived here (each
            // after that lane's earlier ones), so no commit of this launch
            // lands after the CTA has left
            const unsigned long long t0 = tc::globaltimer_ns();
            while (!tc::mbar_try_cluster(bar(B_DONE), 0)) {
                if (tc::globaltimer_ns() - t0 > kDrainNs) {
                    failed = true;
                    raise_abort();
                    break;
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- softmax: warp w holds rows 32 (w % 4) .. +31 of this
        // CTA (its tensor-memory lanes) and key half w / 4 of every tile, so
        // each row is shared by two threads, one per half
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q);
        // Hand a value to the other thread of this row and take its value:
        // each writes its word, the two warps holding the same rows (quarter
        // and quarter + 4) meet at named barrier 1 + quarter, each reads the
        // other's word.  Both warps pass the same sequence of these barriers
        // (one per tile, one per item), so a warp that leaves its role after
        // a failure arrives once at the barrier (at the end of the role): its
        // partner can be held at most at the next one, and checks the abort
        // flag before every later one.  The words are double-buffered by
        // slot: a word is rewritten only after the partner has passed the
        // next barrier, after its read.
        float *xv = xch;  // [slot][half][row]
        auto exchange = [&](int slot, float v, float &other) -> bool {
            if (__any_sync(0xffffffffu, *abort_flag != 0)) {  // one decision for the warp
                failed = true;
                return false;
            }
            xv[(slot * 2 + half) * BM + row] = v;
            asm volatile("bar.sync %0, 64;\n" ::"r"(1 + quarter) : "memory");
            other = xv[(slot * 2 + (half ^ 1)) * BM + row];
            return true;
        };
        for (int i = 0;; i++) {
            ItemInfo it;
            if (!take_item(i, it)) break;
            if (it.stop) break;
            if (it.skip) {
                advance(it);
                continue;
            }
            const int nkt = it.nkt;
            // Without TMA, this CTA's Q rows: 128 rows x 16 chunks, 8 copies
            // per softmax thread.  Every S of the previous item is complete:
            // this thread has been through that item's epilogue, which
            // follows its last PV, which follows its last S.
            if (!p.q_tma) {
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    const int e = tid + kSoftmaxThreads * u;
                    const int r = e >> 4, c = e & 15;
                    const int R = it.row0 + r;
                    const int jr = R / G;
                    const bool ok = jr < it.n;
                    const __nv_bfloat16 *src =
                        ok ? qg + ((size_t)(it.q0 + jr) * p.num_q_heads + it.kvh * G + (R - jr * G)) * D + c * 8 : qg;
                    pkv::cp_async16(smem + kOffQ + (c >> 3) * kQHalf + sw128(r, c & 7), src, ok ? 16 : 0);
                }
                pkv::cp_async_commit();
                pkv::cp_async_wait<0>();
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive_remote(bar_even(B_GO + (go_count & 1)));
            }

            const int R = it.row0 + row;
            const int jrow = R / G;
            const bool row_ok = jrow < it.n;
            // last visible key: causal within the chunk, or the whole shared prefix
            const int pos = !row_ok ? -1 : p.prefix_len ? p.prefix_len - 1 : it.L - it.n + jrow;
            float m_used = -INFINITY, lsum = 0.f;

            bool ok = true;
            for (int t = 0; t < nkt; t++) {
                const int g = g0 + t;
                // S(g) done (the S that read its K stage is done)
                if (!(ok = wait_warp(B_KEMPTY + g % kKStages, (unsigned)((g / kKStages) & 1)))) break;
                tc::fence_after_sync();
                // This thread's 64 scores in one load, whose own reduction
                // gives their maximum; then the buffer is free for S(g+2).
                float sv[64], mp;
                tc::tmem_ld64_max(t_lane + (uint32_t)((g & 1) * BN + half * 64), sv, mp);
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive_remote(bar_even(B_SFREE + (g & 1)));
                const bool full_tile = t * BN + BN <= it.mask_from;
                const int lim0 = pos - t * BN - half * 64;  // this thread's keys i <= lim0 are visible
                if (!full_tile || !row_ok) {
#pragma unroll
                    for (int i2 = 0; i2 < 64; i2++) sv[i2] = i2 <= lim0 ? sv[i2] : -INFINITY;
                    float mx[8];
#pragma unroll
                    for (int i2 = 0; i2 < 8; i2++)
                        mx[i2] = fmaxf(fmaxf(fmaxf(sv[i2], sv[i2 + 8]), fmaxf(sv[i2 + 16], sv[i2 + 24])),
                                       fmaxf(fmaxf(sv[i2 + 32], sv[i2 + 40]), fmaxf(sv[i2 + 48], sv[i2 + 56])));
                    mp = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                }
                if (!row_ok) mp = -INFINITY;
                // P = 2^(s * scale - m) as bf16 pairs over this thread's 64 keys
                // and their sum, against the reference m_used; the scaling runs
                // on paired fp32 multiply-adds
                float pk[32], lt;
                auto compute_p = [&]() {
                    const float nbase = m_used == -INFINITY ? 0.f : -m_used;
                    const uint64_t sc2 = tc::f2(p.scale_log2, p.scale_log2), nb2 = tc::f2(nbase, nbase);
                    // the row sum adds the bf16 values the PV product
                    // multiplies, so that numerator and denominator share
                    // their rounding (a row whose weight sits on one key then
                    // gets that key's V, not V times 1 +- 2^-9): each half of
                    // a packed pair added to an fp32 sum as it stands
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int i2 = 0; i2 < 32; i2++) {
                        float x0, x1;
                        tc::unf2(tc::ffma2(tc::f2(sv[2 * i2], sv[2 * i2 + 1]), sc2, nb2), x0, x1);
                        const uint32_t w = pkv::pack_bf16(tc::ex2(x0), tc::ex2(x1));
                        pk[i2] = __uint_as_float(w);
                        tc::add_bf16_pair(w, acc[(i2 & 1) * 2], acc[(i2 & 1) * 2 + 1]);
                    }
                    lt = (acc[0] + acc[1]) + (acc[2] + acc[3]);
                };
                // the row's maximum over both halves: both threads of the row
                // take the same decisions from here on
                float mo;
                if (!(ok = exchange(g & 1, mp, mo))) break;
                const float mt = fmaxf(mp, mo) * p.scale_log2;  // scale > 0 commutes with max; -inf stays
                const bool need = mt > m_used + 8.f;
                float alpha = 1.f;
                if (need) {
                    alpha = tc::ex2(m_used - mt);  // 0 when nothing was seen yet
                    lsum *= alpha;
                    m_used = mt;
                }
                if (t >= 1 && __any_sync(0xffffffffu, need)) {
                    // rare: rescale this thread's half of the O row once PV(g-1)
                    // is done (O then holds every earlier tile of the item)
                    if (!(ok = wait_warp(B_VEMPTY + (g - 1) % kVStages, (unsigned)(((g - 1) / kVStages) & 1))))
                        break;
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < 64; c += 16) {
                        float o[16];
                        tc::tmem_ld16(t_lane + kOCol + (uint32_t)(half * 64 + c), o);
#pragma unroll
                        for (int i2 = 0; i2 < 16; i2++) o[i2] *= alpha;
                        tc::tmem_st16(t_lane + kOCol + (uint32_t)(half * 64 + c), o);
                    }
                }
                compute_p();
                lsum += lt;
                // P(g)'s buffer was last read by PV(g-2)
                if (g >= 2) {
                    if (!(ok = wait_warp(B_VEMPTY + (g - 2) % kVStages, (unsigned)(((g - 2) / kVStages) & 1))))
                        break;
                    tc::fence_after_sync();
                }
                // keys 64 half .. +63 -> P columns 32 half .. +31 of the buffer,
                // handed to the PV lane once the warp's stores are complete
                tc::tmem_st32(t_lane + kPCol + (uint32_t)((g & 1) * 64 + half * 32), pk);
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive_remote(bar_even(B_PFULL + 2 * (g & 1) + half));
            }
            if (!ok) break;

            // the item's last PV done; the row sum over both halves
            {
                const int gl = g0 + nkt - 1;
                if (!wait_warp(B_VEMPTY + gl % kVStages, (unsigned)((gl / kVStages) & 1))) break;
                tc::fence_after_sync();
            }
            float lo;
            if (!exchange(2 + (go_count & 1), lsum, lo)) break;
            const float ltot = lsum + lo;
            const float inv = ltot > 0.f ? 1.f / ltot : 0.f;
            // Output: each thread writes its half row (columns 64 half ..
            // +63) straight from registers; shared memory stays free for the
            // next item's tiles.
            OutT *orow = static_cast<OutT *>(p.out) +
                         ((size_t)(it.q0 + (row_ok ? jrow : 0)) * p.num_q_heads + it.kvh * G + (R - jrow * G)) * D;
#pragma unroll 1
            for (int c = 0; c < 64; c += 32) {
                float a[32];
                const uint32_t col = (uint32_t)(half * 64 + c);
                tc::tmem_ld32(t_lane + kOCol + col, a);
                if (row_ok && p.prefix_len) {
                    // shared-prefix mode: the unnormalised state (M, L, O)
                    // goes to partial slot 0 of the decode row (s = jrow)
                    const size_t prow = ((size_t)jrow * p.num_q_heads + it.kvh * G + (R - jrow * G)) * p.part_stride;
                    float4 *po = reinterpret_cast<float4 *>(p.part_o + prow * D + col);
#pragma unroll
                    for (int k = 0; k < 8; k++) po[k] = make_float4(a[4 * k], a[4 * k + 1], a[4 * k + 2], a[4 * k + 3]);
                    if (half == 0 && c == 0) *reinterpret_cast<float2 *>(p.part_ml + prow * 2) = make_float2(m_used, ltot);
                } else if (row_ok) {
                    alignas(16) OutT v[32];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) pkv::store2(v + e, a[e] * inv, a[e + 1] * inv);
                    if (p.out_v8) {
                        // 32 bytes per store: each fills whole sectors of the row
                        constexpr int kVec = 32 * (int)sizeof(OutT) / 32;
#pragma unroll
                        for (int k = 0; k < kVec; k++)
                            tc::st_global_32B(orow + col + k * (32 / (int)sizeof(OutT)),
                                              reinterpret_cast<const uint4 *>(v) + 2 * k);
                    } else {
                        constexpr int kVec = 32 * (int)sizeof(OutT) / 16;
#pragma unroll
                        for (int k = 0; k < kVec; k++)
                            reinterpret_cast<uint4 *>(orow + col)[k] = reinterpret_cast<const uint4 *>(v)[k];
                    }
                }
            }
            // the O reads are done before the next item's first PV may overwrite
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_remote(bar_even(B_EPI));
            advance(it);
        }
        if (failed) {
            // the abort flag (raised by whichever wait failed) is visible to
            // the partner warp before it is let past the pending barrier
            *abort_flag = 1;
            __threadfence_block();
            asm volatile("bar.arrive %0, 64;\n" ::"r"(1 + quarter) : "memory");
        }
    }

    pkv::cp_async_wait<0>();
    tc::fence_before_sync();
    const bool any_failed = __syncthreads_or(failed) != 0;
    if (any_failed && tid == 0) {
        pkv::flag(p.status, PKV_STATUS_INTERNAL);
        if (!misaligned) raise_abort();  // the pair takes the same branch below
    }
    tc::cluster_sync();  // both CTAs done with each other's barriers; abort flags final
    // the same decision in both CTAs: every failure raised the abort flag in
    // both, and misaligned shared memory is the pair's (same base)
    if (misaligned || *abort_flag) {
        // copies already issued (by either CTA, counted on the even CTA's
        // barriers) land before either CTA leaves
        const unsigned long long t0 = tc::globaltimer_ns();
        while (tc::globaltimer_ns() - t0 < kGraceNs) {
        }
        tc::cluster_sync();
    }
    tc::fence_after_sync();
    if (warp == 0 && !misaligned) tc::tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

namespace pkv {

bool prefill_tc_supported(int dtype, int head_dim) { return dtype == PKV_BF16 && head_dim == D; }

}  // namespace pkv

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

void encode_once();

// 2-D view of one cache: [num_blocks * num_kv_heads * 16 rows][128 columns]
// bf16, boxes of 16 rows x 64 columns, 128-byte swizzle, zero fill.
int make_cache_map(CUtensorMap *map, const void *cache, int num_blocks, int num_kv_heads) {
    encode_once();
    if (!g_encode) return pkv::fail(PKV_ERR_CUDA, "prefill: cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)num_blocks * num_kv_heads * kBlock};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBlock};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(cache), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return pkv::fail(PKV_ERR_CUDA, "prefill: cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PKV_OK;
}

void encode_once() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
}

// 3-D view of the queries [total_q][Hq][128] bf16: boxes of {64 columns, G
// heads, 128/G queries}, one CTA's 128 packed rows, 128-byte swizzle.
int make_q_map(CUtensorMap *map, const void *q, int num_q_heads, int total_q, int group) {
    encode_once();
    if (!g_encode) return pkv::fail(PKV_ERR_CUDA, "prefill: cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)num_q_heads, (cuuint64_t)total_q};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)num_q_heads * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)(BM / group)};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return pkv::fail(PKV_ERR_CUDA, "prefill: cuTensorMapEncodeTiled (q) failed (%d)", (int)r);
    return PKV_OK;
}

// Per device: the kernel's shared-memory attribute is set (bit 0 float
// output, bit 1 bf16 output) and how many CTA pairs can be resident at once.
// Host threads that race here set the same attribute and store the same count.
std::atomic<unsigned> g_attr_set[64];
std::atomic<int> g_max_pairs[64];

template <typename OutT>
int max_resident_pairs(int dev) {
    int n = dev >= 0 && dev < 64 ? g_max_pairs[dev].load(std::memory_order_relaxed) : 0;
    if (n > 0) return n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, prefill_tc_kernel<OutT>, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) cudaGetLastError();
        n = sms >= 2 ? sms / 2 : 1;
    }
    if (dev >= 0 && dev < 64) g_max_pairs[dev].store(n, std::memory_order_relaxed);
    return n;
}

template <typename OutT>
int launch_typed(const PrefillParams &pp, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                 cudaStream_t st) {
    int dev = 0;
    cudaGetDevice(&dev);
    const unsigned bit = sizeof(OutT) == 4 ? 1u : 2u;
    if (dev >= 0 && dev < 64 && !(g_attr_set[dev].load(std::memory_order_acquire) & bit)) {
        if (cudaFuncSetAttribute(prefill_tc_kernel<OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
            cudaSuccess)
            return pkv::check_launch("prefill_tc: set shared memory size");
        g_attr_set[dev].fetch_or(bit, std::memory_order_acq_rel);
    }
    const int pairs = max_resident_pairs<OutT>(dev);
    // one persistent CTA pair per two SMs (its shared memory allows no second CTA)
    const unsigned grid = 2u * (unsigned)(pp.num_items < pairs ? pp.num_items : pairs);
    prefill_tc_kernel<OutT><<<grid, kThreads, kSmemBytes, st>>>(pp, tq, tk, tv);
    return pkv::check_launch("prefill_tc");
}

}  // namespace

namespace pkv {

void set_wait_limit_ns(unsigned long long ns) { g_wait_ns.store(ns ? ns : kDefaultWaitNs); }

int launch_prefill_tc(const PrefillParams &p, int num_seqs, int out_dtype, cudaStream_t st) {
    if ((long long)p.num_blocks * p.num_kv_heads * kBlock > 0x7fffffffLL)
        return fail(PKV_ERR_INVALID, "prefill: cache too large for 32-bit row coordinates");
    CUtensorMap tk, tv;
    int rc = make_cache_map(&tk, p.k_cache, p.num_blocks, p.num_kv_heads);
    if (rc) return rc;
    rc = make_cache_map(&tv, p.v_cache, p.num_blocks, p.num_kv_heads);
    if (rc) return rc;
    // q tiles by TMA when a CTA's 128 rows are whole queries (G divides 128)
    CUtensorMap tq;
    memset(&tq, 0, sizeof(tq));
    const bool q_tma = p.group <= BM && BM % p.group == 0 && p.total_q > 0;
    if (q_tma) {
        rc = make_q_map(&tq, p.q, p.num_q_heads, p.total_q, p.group);
        if (rc) return rc;
    }
    PrefillParams pp = p;
    pp.q_tma = q_tma ? 1 : 0;
    pp.out_v8 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0 ? 1 : 0;
    pp.num_seqs = num_seqs;
    pp.tiles_per_seq = (p.max_q_len * p.group + kPairRows - 1) / kPairRows;
    pp.wait_ns = g_wait_ns.load();
    const long long items = (long long)num_seqs * p.num_kv_heads * pp.tiles_per_seq;
    if (items > 0x7fff0000LL) return fail(PKV_ERR_INVALID, "prefill: too many q tiles");
    pp.num_items = (int)items;
    if (pp.num_items == 0) return PKV_OK;
    if (reinterpret_cast<uintptr_t>(pp.item_counter) & 15u)
        return fail(PKV_ERR_INVALID, "prefill: the workspace must be 16-byte aligned");
    pp.launch_tag = pkv::next_launch_tag();
    if (pp.launch_tag == 0) pp.launch_tag = 1;  // 0 marks a cleared counter
    return out_dtype == PKV_F32 ? launch_typed<float>(pp, tq, tk, tv, st)
                                : launch_typed<__nv_bfloat16>(pp, tq, tk, tv, st);
}

}  // namespace pkv
