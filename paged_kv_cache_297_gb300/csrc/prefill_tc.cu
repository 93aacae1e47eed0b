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
//   S(t)  = Q K(t)^T : M=256, N=128 keys, K=d; A = Q (each CTA its 128 rows),
//                      B = K (each CTA 64 of the 128 keys), S in each CTA's
//                      tensor memory (its 128 rows x 128 keys);
//   O    += P(t) V(t): M=256, N=d, K=128 keys; A = P from each CTA's tensor
//                      memory, B = V (each CTA 64 of the 128 columns of d).
// One MMA instruction does both SMs' work, and each SM loads only half of
// every K and V tile.  (Measured on GB300: one thread issues a tcgen05.mma
// about every 64 cycles whatever its N, and one thread issues a 2 KB TMA box
// about every 130-180 cycles; the one-SM form of this kernel was bound by the
// latter.)
// Warp roles (one CTA per SM, 12 warps, in both CTAs of the pair):
//   * two softmax teams of 4 warps: team 0 takes key tiles 0, 2, 4, ..., team 1
//     tiles 1, 3, 5, ...  Thread r of a team owns query row r of its CTA
//     (TMEM lane r).  It reads its 128 scores from TMEM in one load, whose
//     own reduction gives the row maximum, masks them, computes
//     p = 2^(s * scale * log2 e - m) (one paired multiply-add per two
//     elements, ex2.approx on the special-function unit) and stores P as bf16
//     pairs over the first 64 columns of the same S buffer, handing each half
//     (64 keys) to its team's MMA lane once both CTAs have stored it.  Each
//     team has its own S/P buffer, O accumulator and running (m, l); the two
//     partial results are merged by log-sum-exp at the end.  One team's
//     softmax overlaps the other team's MMAs.
//   * two MMA-issuing lanes, lane 0 of warps 8 (team 0's tiles) and 9 (team
//     1's) of the even CTA, each in its team's tile order: PV(t) (half by
//     half as P(t) is stored), then S(t+2) into the same buffer.  tcgen05.mma
//     operations issued by one thread execute in order, so S(t+2) cannot
//     overwrite P(t) before PV(t) has read it; the two lanes touch disjoint
//     tensor memory and ring stages, and while one is blocked issuing (the
//     pipe takes an MMA about as fast as it runs one) or waiting for its
//     team's P, the other proceeds.
//   * two loader warps per CTA, one for K and one for V, that gather this
//     CTA's half of each tile through the block table with 2-D TMA boxes (the
//     cache viewed as [num_blocks * num_kv_heads * 16 rows][128] with 128-byte
//     swizzle, which writes exactly the layout the MMAs read), reading the
//     table one tile ahead.  K: this CTA's 4 blocks of the tile's 8, both
//     64-column halves; blocks past the keys are not loaded (their scores are
//     masked).  V: all 8 blocks, this CTA's 64 columns; rows past the keys are
//     zeroed in place (P = 0 times a NaN in an unused row would still poison
//     O) and a block that the keys end inside is copied with zero-filling
//     cp.async.  Every load of either CTA counts its bytes on the even CTA's
//     barrier of that stage, where the MMA lane waits.  Each team has stages
//     of its own in both rings (three for K, two for V), so that every phase
//     of a stage is waited for by one lane, in order; a stage is refilled when
//     the S (for K) or PV (for V) that read it has finished.  The K loader
//     also loads this CTA's Q rows of each item (TMA, 3-D box) and, in the
//     even CTA, hands out the items.
// The running max of a row is only moved when a tile maximum exceeds it by
// more than 8 (log2 units), so P <= 256 and O is rarely rescaled; numerator
// and denominator share the same reference, so the result is exact.
//
// TMEM columns (all 512, in each CTA): S/P of team t at 128t, O of team t at
// 256 + 128t.  Shared memory per CTA, in the 128-byte-swizzled canonical
// layout (8-row atoms of 8 x 128 bytes, 16-byte chunk c of row r at chunk
// c ^ (r % 8)):
//   Q : two 64-column halves of this CTA's 128 rows              (32 KB)
//   K : six stages x two 64-column halves of this CTA's 64 keys  (96 KB)
//   V : four stages x 128 keys of this CTA's 64 columns          (64 KB)
// Waits.  Every wait on an mbarrier is bounded in time (PrefillParams::
// wait_ns, from %globaltimer).  A wait that runs out makes the whole warp
// leave its role loop (the decision is taken warp-wide, so no lane is left
// at a warp barrier) and raises an abort flag in both CTAs, at which the
// other roles' waits give up too.  A role that has left issues no further
// copies or MMAs.  At the end one thread of each CTA waits for the MMA
// thread's final commit, which arrives after every earlier one (a separate,
// fixed bound of one second), the pair meets at a cluster barrier, and if
// anything failed both CTAs wait 100 us more so that copies already issued
// land before either CTA's shared memory is released; the CTA records
// PKV_STATUS_INTERNAL, frees its tensor memory and returns.  (A failure
// stops all further issue, so the only copies that can still be in flight
// were issued before it; a TMA load or cp.async of a few KB lands within
// microseconds.  Waiting on their barriers instead is not possible: after a
// failure a phase may never collect all its arrivals.)
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
constexpr int BM = 128;        // query rows per CTA
constexpr int kPairRows = 256;  // query rows per work item (both CTAs)
constexpr int BN = 128;        // keys per tile
constexpr int kTeamThreads = 128;
constexpr int kMmaWarp = 8;  // warps 8 (team 0) and 9 (team 1) of the even CTA: MMA issue
constexpr int kKLoadWarp = 10, kVLoadWarp = 11;
constexpr int kThreads = 12 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;  // S/P of team t at 128t, O of team t at kOCol + 128t
// Each ring has stages of its own per softmax team: the team's j-th key
// tile goes to stage team * n + j % n of a ring with n stages per team, so
// every phase of a stage is waited for by one issuing thread, in order.  K
// gets three per team: the next S of a team is issued a team period after
// its previous one, about the latency of a K load.
constexpr int kKPerTeam = 3, kVPerTeam = 2;
constexpr int kKStages = 2 * kKPerTeam, kVStages = 2 * kVPerTeam;

constexpr int kQHalf = BM * 128;        // 16 KB: 128 rows x 64 bf16
constexpr int kQBytes = 2 * kQHalf;     // 32 KB
constexpr int kKHalf = 64 * 128;        // 8 KB: this CTA's 64 keys x 64 bf16
constexpr int kKStage = 2 * kKHalf;     // 16 KB
constexpr int kVStage = BN * 128;       // 16 KB: 128 keys x this CTA's 64 bf16
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;                  // 32768
constexpr int kOffV = kOffK + kKStages * kKStage;       // 98304
constexpr int kOffBar = kOffV + kVStages * kVStage;     // 163840

// mbarrier indices.  "both": each CTA has its own, signalled for both by the
// even CTA's MMA commits.  "even": used in the even CTA only, which both
// CTAs' threads (or copies) arrive at.
enum Bar : int {
    B_PFULL = 0,        // [team][half] P(t) of keys 64h .. 64h+63 stored; even, 8 warps
    B_KFULL = 4,        // [stage] K tile landed (both halves); even, 2 loaders + bytes
    // [stage] the S reading the stage is done; both.  Also the softmax
    // team's "S(t) computed" (and, as the MMAs before it are done too, "its
    // PV(t-2) done"): the stage cannot be reused before the team has
    // finished with tile t, so the phase the team waits for is never
    // overtaken
    B_KEMPTY = B_KFULL + kKStages,
    B_VFULL = B_KEMPTY + kKStages,   // [stage] V tile landed; even, 2 loaders + bytes
    // [stage] the PV reading the stage is done; both.  Also the team's "PV(t)
    // done" at the end of an item (same argument)
    B_VEMPTY = B_VFULL + kVStages,
    B_GO = B_VEMPTY + kVStages,      // [k & 1] Q of the k-th item with work landed; even
    B_ITEM_FULL = B_GO + 2,          // [slot] item published; both
    B_ITEM_EMPTY = B_ITEM_FULL + 2,  // [slot] every reader of both CTAs has read it; even
    B_DONE = B_ITEM_EMPTY + 2,       // all MMAs finished (the last commit); both
    B_QFREE = B_DONE + 1,            // every S of the k-th item with work finished; both, 2 commits
    B_EPI = B_QFREE + 1,             // the k-th item's O read by both CTAs' softmax warps; even, 16 warps
    B_ML = B_EPI + 1,                // [team] the team's (m, l) of the k-th item written; per CTA, 4 warps
    kNumBars = B_ML + 2,
};
// item queue readers: even CTA V loader, two MMA lanes and 8 softmax warps;
// odd CTA K loader, V loader and 8 softmax warps
constexpr int kItemReaders = 21;
constexpr int kOffSlots = (kOffBar + kNumBars * 8 + 15) & ~15;  // TMEM address (16 B), two item slots, abort flag
static_assert(kOffSlots % 16 == 0, "item slots are 16-byte vectors");
constexpr int kOffAbort = kOffSlots + 16 + 2 * 16;
constexpr int kOffRed = kOffAbort + 16;
constexpr int kSmemBytes = kOffRed + 2 * 2 * 2 * BM * 4;  // [item & 1][team][m, l][row]
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

// Count this CTA's exit in the second pair of the workspace counter,
// {launch tag, CTAs done}, installed like the first.  The launch's last CTA
// clears both tags, so the next launch installs its own pairs even when it
// carries this launch's tag: a launch replayed from a CUDA graph keeps the
// parameters, tag included, that it was captured with.  (By then every CTA
// has made its last fetch from the first pair.)
__device__ __forceinline__ void count_exit(const PrefillParams &p) {
    const unsigned long long k = pkv::tagged_add(p.item_counter + 2, p.launch_tag);
    if (k == (unsigned long long)gridDim.x - 1) {
        atomicExch(p.item_counter, 0ull);
        atomicExch(p.item_counter + 2, 0ull);
    }
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
    float *red = reinterpret_cast<float *>(smem + kOffRed);  // [item & 1][team][m, l][row]
    // shared::cta address of barrier i, and the shared::cluster windows of
    // the even CTA, this CTA and the other CTA
    auto bar = [&](int i) { return sbase + kOffBar + 8u * (uint32_t)i; };
    const uint32_t base_even = tc::mapa(sbase, 0), base_own = tc::mapa(sbase, rank),
                   base_other = tc::mapa(sbase, rank ^ 1u);
    auto bar_even = [&](int i) { return base_even + kOffBar + 8u * (uint32_t)i; };
    auto bar_own = [&](int i) { return base_own + kOffBar + 8u * (uint32_t)i; };
    auto bar_other = [&](int i) { return base_other + kOffBar + 8u * (uint32_t)i; };

    if (tid == 0 && !misaligned) {
        for (int t = 0; t < 2; t++) {
            tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_PFULL + 2 * t, 8);
            tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_PFULL + 2 * t + 1, 8);
            tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_ITEM_FULL + t, 1);
            tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_ITEM_EMPTY + t, kItemReaders);
            // Q lands by TMA (each CTA's K loader arrives with its bytes) or
            // by the softmax threads' copies (8 warps in each CTA)
            tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_GO + t, p.q_tma ? 2 : 16);
            tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_ML + t, 4);
        }
        tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_DONE, 2);  // one final commit per issuing lane
        tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_QFREE, 2);
        tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_EPI, 16);
        for (int st = 0; st < kKStages; st++) {
            tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_KFULL + st, 2);
            tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_KEMPTY + st, 1);
        }
        for (int st = 0; st < kVStages; st++) {
            tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_VFULL + st, 2);
            tc::mbar_init(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_VEMPTY + st, 1);
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
    auto take_item = [&](int i, ItemInfo &it) -> bool {
        if (!wait_lane0(B_ITEM_FULL + (i & 1), (unsigned)((i >> 1) & 1))) return false;
        const int4 v = item_slots[i & 1];
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_cluster(bar_even(B_ITEM_EMPTY + (i & 1)));
        it = item_info(p, v, rank);
        return true;
    };

    // Running counts that carry the barrier phases from one item to the next:
    // tiles of each team (its ring stages and P barriers) and items with work
    // (the Q, epilogue and (m, l) barriers).  Every role of both CTAs walks
    // the same items, so every role's counts agree.
    int team_base0 = 0, team_base1 = 0, go_count = 0;
    auto advance = [&](const ItemInfo &it) {
        team_base0 += (it.nkt + 1) / 2;
        team_base1 += it.nkt / 2;
        go_count += it.skip ? 0 : 1;
    };

    // Ring slot of tile t of the current item: the team's j-th tile goes to
    // stage team * n + j % n, phase j / n of that stage's barriers (n stages
    // per team: kKPerTeam for K, kVPerTeam for V).
    auto team_tile = [&](int t) { return ((t & 1) ? team_base1 : team_base0) + (t >> 1); };
    auto kstage = [&](int t) { return (t & 1) * kKPerTeam + team_tile(t) % kKPerTeam; };
    auto kphase = [&](int t) { return (unsigned)((team_tile(t) / kKPerTeam) & 1); };
    auto vstage = [&](int t) { return (t & 1) * kVPerTeam + team_tile(t) % kVPerTeam; };
    auto vphase = [&](int t) { return (unsigned)((team_tile(t) / kVPerTeam) & 1); };

    if (failed) {
        // nothing: misaligned shared memory (reported below)
    } else if (warp == kKLoadWarp || warp == kVLoadWarp) {
        // ---------------- loaders; the even CTA's K loader also runs the item queue
        const bool is_k = warp == kKLoadWarp;
        const CUtensorMap *tmap_kv[2] = {&tmap_k, &tmap_v};
        const int full0 = is_k ? B_KFULL : B_VFULL, empty0 = is_k ? B_KEMPTY : B_VEMPTY;
        const unsigned char *cache = static_cast<const unsigned char *>(is_k ? p.k_cache : p.v_cache);
        int item = (int)(blockIdx.x >> 1);  // the cluster's first item; later ones come from the counter
        for (int i = 0;; i++) {
            ItemInfo it;
            if (is_k && even) {
                int4 v = make_int4(item, 0, 0, 0);
                if (i >= 2 && !wait_lane0(B_ITEM_EMPTY + (i & 1), (unsigned)(((i >> 1) - 1) & 1))) break;
                if (lane == 0) {
                    if (item < p.num_items && p.prefix_len) {
                        v.y = 0;                // the decode queries, one "position" per sequence
                        v.z = p.max_q_len;
                        v.w = p.prefix_len;
                    } else if (item < p.num_items) {
                        const int s = p.num_seqs - 1 - item / (p.num_kv_heads * p.tiles_per_seq);
                        v.y = p.cu_q_lens[s];
                        v.z = p.cu_q_lens[s + 1] - v.y;
                        v.w = p.context_lens[s];
                    }
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
            if (is_k && p.q_tma && !it.skip) {
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
            const int nb = is_k ? 4 : 8;              // blocks of a tile this CTA loads
            const int b0 = is_k ? 4 * (int)rank : 0;  // the first of them
            // Block ids of this CTA's blocks of tile t (lane q < nb: block q),
            // -1 past the keys.  They are read one tile ahead, so the copies
            // of a tile never wait for its table entries.
            auto table_id = [&](int t) {
                int id = -1;
                if (t < it.nkt && lane < nb && t * BN + (b0 + lane) * kBlock < it.kv_end) id = table[t * 8 + b0 + lane];
                return id;
            };
            int next_id = table_id(0);
            bool ok = true;
            for (int t = 0; t < it.nkt; t++) {
                const int per = is_k ? kKPerTeam : kVPerTeam;
                const int st = is_k ? kstage(t) : vstage(t), jt = team_tile(t);
                // the stage's previous tile (the team's tile jt - per) has been read
                if (jt >= per && !(ok = wait_warp(empty0 + st, (unsigned)((jt / per - 1) & 1)))) break;
                const int my_id = next_id;
                next_id = table_id(t + 1);
                const uint32_t full = bar_even(full0 + st);
                const int tile_keys = min(BN, it.kv_end - t * BN);
                const int nbk = (tile_keys + kBlock - 1) / kBlock;  // blocks of the tile holding keys
                const int box_rows = p.num_blocks * p.num_kv_heads * kBlock;  // rows of the 2-D view
                if (is_k) {
                    // this CTA's keys: blocks 4*rank .. 4*rank+3 of the tile,
                    // those holding keys (the rest are masked out of S)
                    unsigned char *dst = smem + kOffK + st * kKStage;
                    const int nk = max(0, min(4, nbk - 4 * (int)rank));
                    int y = box_rows;
                    if (lane < nk) {
                        if (my_id >= 0 && my_id < p.num_blocks)
                            y = (my_id * p.num_kv_heads + it.kvh) * kBlock;
                        else
                            pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                    }
                    int ys[4];
#pragma unroll
                    for (int q = 0; q < 4; q++) ys[q] = __shfl_sync(0xffffffffu, y, q);
                    if (lane == 0) {
                        tc::mbar_arrive_expect_tx_remote(full, (uint32_t)(nk * 2 * 2048));
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            if (q >= nk) break;
#pragma unroll
                            for (int h = 0; h < 2; h++)
                                tc::tma_load_2d_pair(dst + h * kKHalf + q * 2048, tmap_kv[0], h * 64, ys[q], full);
                        }
                    }
                } else {
                    // all 8 blocks, this CTA's 64 columns of d; a block that
                    // the keys end inside by zero-filling copies, rows past
                    // the keys zeroed
                    unsigned char *dst = smem + kOffV + st * kVStage;
                    const int cpq = (tile_keys % kBlock) ? tile_keys / kBlock : -1;
                    const int ntma = cpq >= 0 ? nbk - 1 : nbk;  // blocks 0 .. ntma-1 by TMA
                    int y = box_rows;
                    if (lane < ntma) {
                        if (my_id >= 0 && my_id < p.num_blocks)
                            y = (my_id * p.num_kv_heads + it.kvh) * kBlock;
                        else
                            pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                    }
                    int ys[8];
#pragma unroll
                    for (int q = 0; q < 8; q++) ys[q] = __shfl_sync(0xffffffffu, y, q);
                    if (cpq >= 0 || nbk < 8) {
                        // generic-proxy part of the tile: the partial block's
                        // live rows by zero-filling copies, every other row
                        // past the keys zeroed with stores
                        const int phys = cpq >= 0 ? __shfl_sync(0xffffffffu, my_id, cpq) : 0;
                        const bool bok = phys >= 0 && phys < p.num_blocks;
                        if (cpq >= 0 && !bok && lane == 0) pkv::flag(p.status, PKV_STATUS_BAD_BLOCK);
                        for (int e = lane + 16 * 8 * ntma; e < BN * 8; e += 32) {
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
                        tc::mbar_arrive_expect_tx_remote(full, (uint32_t)(ntma * 2048));
#pragma unroll
                        for (int q = 0; q < 8; q++) {
                            if (q >= ntma) break;
                            tc::tma_load_2d_pair(dst + q * 2048, tmap_kv[1], (int)rank * 64, ys[q], full);
                        }
                    }
                }
            }
            if (!ok) break;
            advance(it);
            if (is_k && even) {  // the next item, fetched while the consumers work on this one
                if (lane == 0) item = next_item(p);
                item = __shfl_sync(0xffffffffu, item, 0);
            }
        }
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
        // ---------------- MMA issue: lane 0 of warp 8 (team 0's tiles) and of
        // warp 9 (team 1's tiles) of the even CTA issue every MMA of the
        // pair.  The two lanes touch disjoint tensor memory (each team's S/P
        // buffer and O accumulator) and disjoint ring stages, and each
        // lane's MMAs run in its issue order, so neither needs to order
        // itself after the other: while one is blocked issuing into the
        // tensor pipe (which takes an MMA about as fast as it runs it) or
        // waiting for its team's P, the other's waits and commits proceed.
        const int team = warp - kMmaWarp;
        if (even && lane == 0) {
            // one commit per CTA of the pair: each CTA's barrier i
            auto commit_both = [&](int i) {
                tc::mma_commit_pair(bar_own(i));
                tc::mma_commit_pair(bar_other(i));
            };
            // Descriptors of the first 16 columns of Q and of stage 0 of the K
            // and V rings; a stage, a half or 16 more columns is a constant
            // number of 16-byte units on.  V is MN-major: the next 8 keys at
            // +1 KB (SBO); this CTA's 64 columns are one 128-byte swizzle
            // span (LBO unused).
            const uint64_t q_desc = tc::smem_desc_sw128(sbase + kOffQ, 16, 1024);
            const uint64_t k_desc0 = tc::smem_desc_sw128(sbase + kOffK, 16, 1024);
            const uint64_t v_desc0 = tc::smem_desc_sw128(sbase + kOffV, kVStage, 1024);
            int nkt_cur = 0;  // key tiles of the item being issued
            // S(t) = Q K(t)^T into this team's S/P buffer (K(t) landed)
            auto issue_s = [&](int t) {
                const int st = kstage(t);
                tc::mma_s_tile_pair<kQHalf / 16, kKHalf / 16>(tmem + team * BN, q_desc,
                                                               k_desc0 + (uint64_t)(st * (kKStage / 16)), kIdescS);
                commit_both(B_KEMPTY + st);
                // the item's last two S (one per lane) are the last reads of
                // Q: the Q barrier expects two arrivals per item
                if (t + 2 >= nkt_cur) commit_both(B_QFREE);
            };
            // O(team) (+)= P(t) V(t) over keys 64h .. 64h+63 (V(t) landed,
            // that half of P(t) stored in both CTAs)
            auto issue_pv_half = [&](int t, int h) {
                const int st = vstage(t);
                tc::mma_pv_half_pair<2048 / 16>(tmem + kOCol + team * D, tmem + team * BN + h * 32,
                                                v_desc0 + (uint64_t)(st * (kVStage / 16) + h * 4 * (2048 / 16)),
                                                kIdescPV, (t < 2 && h == 0) ? 0u : 1u);
                if (h == 1) commit_both(B_VEMPTY + st);
            };
            for (int i = 0;; i++) {
                // Take item i alone (the other lanes idle).  The slot is
                // reported read only after this item's Q barrier has been
                // waited for: the queue then cannot run two items ahead of
                // this lane, so neither Q barrier can complete a phase that
                // this lane has not yet waited for.
                if (!wait1(B_ITEM_FULL + (i & 1), (unsigned)((i >> 1) & 1))) { failed = true; break; }
                const ItemInfo it = item_info(p, item_slots[i & 1], rank);
                if (!it.stop && !it.skip && !wait1(B_GO + (go_count & 1), (unsigned)((go_count >> 1) & 1))) {
                    failed = true;
                    break;
                }
                tc::mbar_arrive_cluster(bar_own(B_ITEM_EMPTY + (i & 1)));
                if (it.stop) break;
                if (!it.skip) {
                    const int nkt = it.nkt;
                    nkt_cur = nkt;
                    if (nkt == 1 && team == 1) {  // one S reads this Q, and it is team 0's
                        tc::mbar_arrive_remote(bar_own(B_QFREE));
                        tc::mbar_arrive_remote(bar_other(B_QFREE));
                    }
                    if (team < nkt) {
                        if (!wait1(B_KFULL + kstage(team), kphase(team))) { failed = true; break; }
                        tc::fence_after_sync();
                        issue_s(team);
                    }
                    // The previous item's O has been read by both CTAs before
                    // this item's first PV overwrites it.
                    if (go_count > 0 && !wait1(B_EPI, (unsigned)((go_count - 1) & 1))) { failed = true; break; }
                    // This team's tiles in order: PV(t) half by half as P(t)
                    // is stored, then S(t+2) into the same buffer once K(t+2)
                    // has landed.
                    const int tb = team ? team_base1 : team_base0;  // the team's tiles before this item
                    for (int t = team; t < nkt && !failed; t += 2) {
                        if (!wait1(B_VFULL + vstage(t), vphase(t))) { failed = true; break; }
                        for (int h = 0; h < 2 && !failed; h++) {
                            if (!wait1(B_PFULL + 2 * team + h, (unsigned)((tb + (t >> 1)) & 1))) {
                                failed = true;
                                break;
                            }
                            tc::fence_after_sync();
                            issue_pv_half(t, h);
                        }
                        if (!failed && t + 2 < nkt) {
                            if (!wait1(B_KFULL + kstage(t + 2), kphase(t + 2))) { failed = true; break; }
                            tc::fence_after_sync();
                            issue_s(t + 2);
                        }
                    }
                    if (failed) break;
                }
                advance(it);
            }
            if (failed) raise_abort();
            // every MMA of this lane has finished, and every earlier commit
            // of it has arrived at this CTA's barriers, before the tensor
            // memory is released
            commit_both(B_DONE);
        }
        if (warp == kMmaWarp && lane == 0) {
            // in both CTAs: both lanes' final commits have arrived here (each
            // after that lane's earlier ones), so no commit of this launch
            // lands after the CTA has left
            const unsigned long long t0 = tc::globaltimer_ns();
            while (!tc::mbar_try_cluster(bar(B_DONE), 0)) {
                if (tc::globaltimer_ns() - t0 > kDrainNs) {
                    failed = true;
                    break;
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- softmax teams
        const int team = warp >> 2, quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t s_col = (uint32_t)team * BN, o_col = kOCol + (uint32_t)team * D;
        const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q);
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
            // per softmax thread.  The previous item's S MMAs are all
            // complete: this thread has been through that item's epilogue,
            // which follows both teams' last PV.
            if (!p.q_tma) {
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    const int e = tid + 2 * kTeamThreads * u;
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
            for (int t = team; t < nkt; t += 2) {
                // S(t) done (the S that read its K stage is done); the team's
                // PV(t-2), issued before it by the same lane, is done too
                if (!(ok = wait_warp(B_KEMPTY + kstage(t), kphase(t)))) break;
                tc::fence_after_sync();
                const bool full_tile = t * BN + BN <= it.mask_from;
                const int lim0 = pos - t * BN;  // keys i <= lim0 of this tile are visible
                // The row's 128 scores in one load, whose own reduction gives
                // their maximum; masked tiles take it from the masked values.
                // P is computed from these registers, and each score register
                // is free once its P is packed.
                const bool masked = !full_tile || !row_ok;
                float sv[BN], mraw;
                tc::tmem_ld128_max(t_lane + s_col, sv, mraw);
                if (masked) {
#pragma unroll
                    for (int i2 = 0; i2 < BN; i2++) sv[i2] = i2 <= lim0 ? sv[i2] : -INFINITY;
                    float mx[16];
#pragma unroll
                    for (int i2 = 0; i2 < 16; i2++)
                        mx[i2] = fmaxf(fmaxf(fmaxf(sv[i2], sv[i2 + 16]), fmaxf(sv[i2 + 32], sv[i2 + 48])),
                                       fmaxf(fmaxf(sv[i2 + 64], sv[i2 + 80]), fmaxf(sv[i2 + 96], sv[i2 + 112])));
#pragma unroll
                    for (int i2 = 0; i2 < 8; i2++) mx[i2] = fmaxf(mx[i2], mx[i2 + 8]);
#pragma unroll
                    for (int i2 = 0; i2 < 4; i2++) mx[i2] = fmaxf(mx[i2], mx[i2 + 4]);
                    mraw = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                }
                if (!row_ok) mraw = -INFINITY;
                const float mt = mraw * p.scale_log2;  // scale > 0 commutes with max; -inf stays
                const bool need = mt > m_used + 8.f;
                float alpha = 1.f;
                if (need) {
                    alpha = tc::ex2(m_used - mt);  // 0 when nothing was seen yet
                    lsum *= alpha;
                    m_used = mt;
                }
                if (t >= 2 && __any_sync(0xffffffffu, need)) {
                    // rare: rescale the team's O (16 columns at a time beside
                    // the scores held in registers)
#pragma unroll 1
                    for (int c = 0; c < D; c += 16) {
                        float o[16];
                        tc::tmem_ld16(t_lane + o_col + c, o);
#pragma unroll
                        for (int i2 = 0; i2 < 16; i2++) o[i2] *= alpha;
                        tc::tmem_st16(t_lane + o_col + c, o);
                    }
                }
                // P = 2^(s * scale - m) as bf16 pairs over the first 64 columns;
                // the scaling and the row sum run on paired fp32 instructions
                const float nbase = m_used == -INFINITY ? 0.f : -m_used;
                const uint64_t sc2 = tc::f2(p.scale_log2, p.scale_log2), nb2 = tc::f2(nbase, nbase);
                uint64_t acc2[2] = {tc::f2(0.f, 0.f), tc::f2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < BN; c += 64) {
                    float pk[32];
#pragma unroll
                    for (int i2 = 0; i2 < 32; i2++) {
                        float x0, x1;
                        tc::unf2(tc::ffma2(tc::f2(sv[c + 2 * i2], sv[c + 2 * i2 + 1]), sc2, nb2), x0, x1);
                        const float e0 = tc::ex2(x0), e1 = tc::ex2(x1);
                        acc2[i2 & 1] = tc::fadd2(acc2[i2 & 1], tc::f2(e0, e1));
                        pk[i2] = __uint_as_float(pkv::pack_bf16(e0, e1));
                    }
                    // keys c .. c+63 -> P columns c/2 .. c/2+31, handed to the
                    // MMA lane once the warp's stores are complete
                    tc::tmem_st32(t_lane + s_col + c / 2, pk);
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive_remote(bar_even(B_PFULL + 2 * team + c / 64));
                }
                {
                    float a0, a1, b0, b1;
                    tc::unf2(acc2[0], a0, a1);
                    tc::unf2(acc2[1], b0, b1);
                    lsum += (a0 + a1) + (b0 + b1);
                }
            }
            if (!ok) break;

            // merge the two teams: exchange (m, l) with the other team's thread
            // of the same row through shared memory (double-buffered by item)
            const int my_tiles = nkt > team ? (nkt - team + 1) / 2 : 0;
            if (my_tiles > 0) {  // the team's last PV done (the PV that read its V stage)
                const int tl = team + 2 * (my_tiles - 1);
                if (!wait_warp(B_VEMPTY + vstage(tl), vphase(tl))) break;
                tc::fence_after_sync();
            }
            float *rb = red + (go_count & 1) * (2 * 2 * BM);
            rb[(team * 2 + 0) * BM + row] = m_used;
            rb[(team * 2 + 1) * BM + row] = lsum;
            // The fences order this thread's later reads of both teams' O
            // after the completion the other team observed; without them the
            // first tcgen05.ld waits microseconds.
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(reinterpret_cast<uint64_t *>(smem + kOffBar) + B_ML + team);
            if (!wait_warp(B_ML + (team ^ 1), (unsigned)(go_count & 1))) break;
            tc::fence_after_sync();
            const float m0 = rb[0 * BM + row], l0 = rb[1 * BM + row];
            const float m1 = rb[2 * BM + row], l1 = rb[3 * BM + row];
            const float M = fmaxf(m0, m1);
            const float f0 = M == -INFINITY ? 0.f : tc::ex2(m0 - M);
            const float f1 = (M == -INFINITY || nkt < 2) ? 0.f : tc::ex2(m1 - M);
            const float ltot = l0 * f0 + l1 * f1;
            const float inv = ltot > 0.f ? 1.f / ltot : 0.f;
            const float g0 = f0 * inv, g1 = f1 * inv;
            // Output: each thread writes its half row (team 0 columns 0..63,
            // team 1 columns 64..127) straight from registers, 16 bytes at a
            // time; shared memory stays free for the next item's tiles.
            OutT *orow = static_cast<OutT *>(p.out) +
                         ((size_t)(it.q0 + (row_ok ? jrow : 0)) * p.num_q_heads + it.kvh * G + (R - jrow * G)) * D;
#pragma unroll 1
            for (int c = 0; c < D / 2; c += 32) {
                float a[32], b[32];
                const uint32_t col = (uint32_t)(team * (D / 2) + c);
                tc::tmem_ld32(t_lane + kOCol + col, a);
                if (nkt >= 2) {
                    tc::tmem_ld32(t_lane + kOCol + D + col, b);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e++) b[e] = 0.f;
                }
                if (row_ok && p.prefix_len) {
                    // shared-prefix mode: the unnormalised state (M, L, O)
                    // goes to partial slot 0 of the decode row (s = jrow)
                    const size_t prow = ((size_t)jrow * p.num_q_heads + it.kvh * G + (R - jrow * G)) * p.part_stride;
                    float4 *po = reinterpret_cast<float4 *>(p.part_o + prow * D + col);
#pragma unroll
                    for (int k = 0; k < 8; k++)
                        po[k] = make_float4(a[4 * k] * f0 + b[4 * k] * f1, a[4 * k + 1] * f0 + b[4 * k + 1] * f1,
                                            a[4 * k + 2] * f0 + b[4 * k + 2] * f1, a[4 * k + 3] * f0 + b[4 * k + 3] * f1);
                    if (team == 0 && c == 0) *reinterpret_cast<float2 *>(p.part_ml + prow * 2) = make_float2(M, ltot);
                } else if (row_ok) {
                    alignas(16) OutT v[32];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) pkv::store2(v + e, a[e] * g0 + b[e] * g1, a[e + 1] * g0 + b[e + 1] * g1);
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
    }

    pkv::cp_async_wait<0>();
    tc::fence_before_sync();
    const bool any_failed = __syncthreads_or(failed) != 0;
    if (any_failed && tid == 0) pkv::flag(p.status, PKV_STATUS_INTERNAL);
    tc::cluster_sync();  // both CTAs done with each other's barriers; abort flags final
    if (*abort_flag || any_failed) {
        // copies already issued (by either CTA, counted on the even CTA's
        // barriers) land before either CTA leaves
        const unsigned long long t0 = tc::globaltimer_ns();
        while (tc::globaltimer_ns() - t0 < kGraceNs) {
        }
    }
    tc::cluster_sync();
    tc::fence_after_sync();
    if (warp == 0 && !misaligned) tc::tmem_dealloc_pair(tmem, kTmemCols);
    // every role of the pair has passed its last item fetch
    if (tid == 0) count_exit(p);
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
