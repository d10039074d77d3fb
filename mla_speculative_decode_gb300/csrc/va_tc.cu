// va_tc.cu -- split-K partial kernel on the tcgen05 tensor cores (K1, TC path).
//
// The step is two dense contractions over a shared latent row (The Milestone
// Commit, "Input Knowledge Required": the draft tokens attend the full KV
// cache; every head reads the same MLA latent row): S = Q K^T over 576
// columns and O = P V over 512, with R = T*H rows per request.  On GB300 the
// accumulator of one 128-row block, O = 128 x 512 fp32, fills a whole SM's
// tensor memory (512 columns), so the QK and the PV products of a row block
// run on two SMs.  A (split, row unit) runs on one cluster, in one of two
// shapes (the kernel template's `kPair`):
//
//   one-SM products (cluster of 2, units of 128 rows): rank 0 is the QK CTA
//     and rank 1 the PV CTA, each issuing its own 128-row products
//     (cta_group::1).
//   two-SM products (cluster of 4, units of 256 rows): ranks 0-1 are a QK
//     pair and ranks 2-3 a PV pair.  The even rank of each pair issues
//     products of M = 256 rows for both (cta_group::2).  Each CTA holds its
//     own 128 rows of the A operand and of the accumulator, and half of the
//     B operand: keys 0-31 or 32-63 of a key tile (all 576 columns); value
//     column blocks {0,1,4,5} or {2,3,6,7} (64 columns each) of a value tile.
//     So each SM gathers half of a tile's bytes per 128 rows, which is what
//     bounds the tile time on paged pools.  The odd rank's MMA warp forwards
//     its tiles' arrivals to the even rank.
//
//   QK CTA (one per 128 rows)
//     TMEM: Q as the A operand (128 lanes x 288 columns of bf16 pairs) and two
//     64-column S buffers.  Warps 0, 2, 3, 12-15 bring the CTA's keys of each
//     64-key tile into a ring of 184 KB (one 64-column block of its keys per
//     slot) in the 128B-swizzled K-major layout (16-byte cp.async gathers for
//     paged keys, TMA boxes for contiguous ones); warp 1 issues S = Q K^T (36
//     MMAs of M x 64 x 16, A from TMEM, B K-major) with two commits per tile
//     (the blocks whose slots the producers refill next, then S ready); warps
//     4-11 are two softmax warpgroups, each owning 32 of a tile's 64 columns
//     for every row: they share the tile maximum through shared memory, run an
//     online softmax with a conditional rescale (the reference max only moves
//     when a tile exceeds it by 2^8), round P to bf16 into a local staging
//     buffer, and one thread ships P with the rows' rescale factors to the PV
//     CTA of the same rows with a single distributed-shared-memory bulk copy
//     into a ring of three P buffers.
//   PV CTA (one per 128 rows)
//     TMEM: O (128 lanes x 512 columns fp32).  Warps 0, 2, 3, 12-15 bring its
//     value columns of the same tiles -- L2 hits behind the QK CTAs' reads --
//     into a ring of 20 slots of 8 KB; warp 1 issues O += P V (8 MMAs of M x
//     256 x 16, A = P K-major, B = V MN-major: the same swizzled block layout
//     is K-major for S and MN-major for PV); warps 4-11 rescale O rows on the
//     rare tiles whose reference max moved, then normalise and write the
//     split's partial, each warpgroup for 256 of the 512 columns.
//
// The design follows the pages' split-K / online-softmax / partial-reduce
// structure (The Milestone Commit, "The Thinking Process Revealed"; The Commit
// That Locked In 6x Decode, "Input Knowledge Required"), moved onto tcgen05,
// TMEM and distributed shared memory.  Every wait is bounded: on timeout the
// CTA sets VA_STATUS_TIMEOUT, stops, drains its own copies and MMAs, frees its
// tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include "va_common.cuh"
#include "va_sm100.cuh"

#ifdef VA_TRACE
__device__ unsigned long long* g_va_trace = nullptr;
extern "C" __attribute__((visibility("default"))) int va_trace_set(void* buf) {
  return cudaMemcpyToSymbol(g_va_trace, &buf, sizeof(buf)) == cudaSuccess ? 0 : -1;
}
#endif

#ifdef VA_TEST_HOOKS
// Test build only (libverifyattn_testhooks.so): a gate that the producer
// warps of every split-K CTA wait on, bounded like every other wait, before
// their first copy.  A test points it at a device flag that nothing sets, so
// the wait runs out, and checks that the kernel gives up cleanly: status
// VA_STATUS_TIMEOUT, every role leaves through its abort path, and the next
// call on the stream is correct.  NULL (the default) = no gate.
__device__ const int32_t* g_va_test_gate = nullptr;
extern "C" __attribute__((visibility("default"))) int va_test_set_gate(const int32_t* flag) {
  return cudaMemcpyToSymbol(g_va_test_gate, &flag, sizeof(flag)) == cudaSuccess ? VA_OK
                                                                               : VA_ERR_CUDA;
}
#endif

namespace va {
namespace {

using namespace sm100;

constexpr int kThreads = 512;
constexpr int kRows = 128;                                  // rows of one CTA
constexpr int kTile = 64;                                   // keys per tile
constexpr int kKBlocks = kDqk / 64;                         // 9 column blocks (K)
constexpr int kVBlocks = kDv / 64;                          // 8 column blocks (V)
constexpr uint32_t kVSlotBytes = kTile * 128;               // 8 KB: 64 keys x 64 value cols
// Value ring: 20 slots of 8 KB, one column block of a 64-key tile per slot
// (tile t's j-th block in slot (nb*t + j) mod 20, nb the blocks a CTA holds).
// Each slot has its own release barrier, committed after the products that
// read it, so the next tiles start loading while the current tile's products
// are still running.  The ring size is a multiple of 4 so that the blocks of
// one PV product (its N extent, 256 or 128 columns per CTA) sit in adjacent
// slots: with A = P read from shared memory, a 256-wide product reads 12 KB of
// shared memory per 128 cycles, a 128-wide one 8 KB per 64 cycles, more than
// the shared memory can deliver next to the incoming copies.
constexpr int kRingV = 20;
// P buffer: P tile (128 rows x 64 keys bf16, K-major 128B swizzle), then the
// rows' rescale factors, then the four softmax warps' rescale flags.  Shipped
// to the PV CTA as one contiguous bulk copy.
constexpr uint32_t kPBytes = kRows * 128;                   // 16 KB
constexpr uint32_t kPAlpha = kPBytes;                       // float [128]
constexpr uint32_t kPFlags = kPAlpha + 4 * kRows;           // uint32 [4]
constexpr uint32_t kPPayload = kPFlags + 16;                // bytes copied
constexpr uint32_t kPBufBytes = 17 * 1024;                  // buffer stride (1024-aligned)
constexpr int kPBufs = 3;                                   // P ring depth (PV CTA)
constexpr uint32_t kCmdDone = 0xFFFFFFFFu;

// The two cluster shapes.  Key ring: 184 KB of slots holding one 64-column
// block of a CTA's keys of a tile (64 keys, 8 KB, or 32 keys, 4 KB, in a
// pair); tile t's block c sits at ring position 9t + c.  Tile t's slots last
// held block kKRelease of tile t - kKLag and the blocks before it (and
// earlier tiles): the QK products commit once after block kKRelease of every
// tile (one release barrier per tile, a ring of kKEmptyRing), and producer 0
// waits for that one commit before filling a tile.  Tiles 1 .. kKLag-1 find
// their slots unused, but the row block's Q lands there at the start (see
// kOffQ) and stays until it is in TMEM.
template <bool kPair>
struct Cfg {
  static constexpr int kCtas = kPair ? 4 : 2;
  static constexpr int kUnitRows = kPair ? 2 * kRows : kRows;
  static constexpr int kSlotKeys = kPair ? kTile / 2 : kTile;   // keys a QK CTA holds per tile
  static constexpr uint32_t kKSlotBytes = uint32_t(kSlotKeys) * 128u;
  static constexpr int kRingK = kPair ? 46 : 23;
  static constexpr int kKLag = kPair ? 5 : 2;
  static constexpr int kKRelease = kPair ? 7 : 3;
  static_assert(kRingK == kKBlocks * kKLag - kKRelease + kKBlocks - 1, "key ring release point");
  static constexpr int kKEmptyRing = kPair ? 8 : 2;
  // Producers run at most kKLag key tiles (value: kRingV / blocks tiles)
  // ahead of the products, so a ring of kFullRing tile-landed barriers is
  // never two phases ahead of its waiter.
  static constexpr int kFullRing = kPair ? 8 : 2;
  static constexpr int kVBlocksCta = kPair ? kVBlocks / 2 : kVBlocks;
  static constexpr int kVGroup = kPair ? 2 : 4;             // value blocks per CTA per product
  // key-validity masks: the producers run at most kKLag tiles ahead of the
  // products and those at most two ahead of the softmax warps
  static constexpr int kValidRing = kPair ? 16 : 8;
  // (producers at tile t follow the commit of tile t - kKLag; the products
  // follow the softmax by at most two tiles)
  static_assert(kValidRing >= kKLag + 2 && kFullRing >= kKLag && kKEmptyRing >= kKLag, "rings");
  static_assert(kRingV % 4 == 0 && kRingV / kVBlocksCta < kFullRing + 1, "value ring");
  static constexpr uint16_t kQkMask = kPair ? 0x3 : 0x1;    // cluster ranks of the QK CTAs
  static constexpr uint16_t kPvMask = kPair ? 0xC : 0x2;

  // Barriers.  The layout is identical in every CTA of the cluster so that
  // remote arrivals and multicast commits land on the right objects.  Names
  // ending in P exist in pairs only: arrivals from the odd rank, forwarded to
  // the even rank that issues the products (PV: a value tile and its P
  // buffer together, one forwarded arrival per tile).
  static constexpr int B_FULL = 0;                          // [kFullRing] tile landed
  static constexpr int B_FULLP = B_FULL + kFullRing;        // [kFullRing] odd rank's tile landed
  static constexpr int B_EMPTY = B_FULLP + (kPair ? kFullRing : 0);
  // B_EMPTY: QK, [kKEmptyRing] key slots of tile t released (t % kKEmptyRing);
  //          PV, [kRingV] value slot released
  static constexpr int kEmpty = kRingV > kKEmptyRing ? kRingV : kKEmptyRing;
  static constexpr int B_SFULL = B_EMPTY + kEmpty;          // [2]
  static constexpr int B_SEMPTY = B_SFULL + 2;              // [2]
  static constexpr int B_PFREE = B_SEMPTY + 2;              // [kPBufs] QK; committed by PV
  static constexpr int B_PFULL = B_PFREE + kPBufs;          // [kPBufs] PV; bulk copies from QK
  static constexpr int B_QREADY = B_PFULL + kPBufs;
  static constexpr int B_QREADYP = B_QREADY + 1;
  static constexpr int B_MMAFIN = B_QREADYP + (kPair ? 1 : 0);
  static constexpr int B_OGO = B_MMAFIN + 1;
  static constexpr int B_OCORR = B_OGO + 1;
  static constexpr int B_ODONE = B_OCORR + 1;
  static constexpr int B_FIN = B_ODONE + 1;
  static constexpr int B_VREADY = B_FIN + 1;                // [kValidRing] key-validity masks
  static constexpr int B_QTMA = B_VREADY + kValidRing;      // Q rows landed (QK)
  static constexpr int kNumBars = B_QTMA + 1;

  // shared layout (offsets from a 1024-byte aligned base)
  static constexpr uint32_t kOffBars = 0;
  static constexpr uint32_t kOffTmemSlot = kPair ? 640 : 512;
  static constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
  static constexpr uint32_t kOffCmd = kOffTmemSlot + 8;     // PV: row-warp command word
  static constexpr uint32_t kOffFlags = kOffTmemSlot + 12;  // uint32: this CTA's status bits
  static constexpr uint32_t kOffValid = kPair ? 704 : 576;  // QK: uint64 [kValidRing]
  static constexpr uint32_t kOffPar = 1024;                 // QK: int32 [64] tree parents
  static constexpr uint32_t kOffFin = 1024;                 // PV: float [128] 1 / row sum
  static constexpr uint32_t kOffSrow = 1536;                // int32 [2][64] staged pool rows
  static constexpr uint32_t kOffMx = 2048;                  // QK: float [2][128] half maxima
  static constexpr uint32_t kOffPeerAny = 2048;             // PV pair, even rank: uint32 [kPBufs]
  static constexpr uint32_t kOffK = 4096;                   // QK: K ring
  static constexpr uint32_t kOffStage = kOffK + kRingK * kKSlotBytes;   // QK: P staging [2]
  // QK: the row block's Q (128 rows x 576 features, two boxes of 64 rows
  // laid out [column block][row][128 B], 128B-swizzled), loaded once at the
  // start past the first tile's slots (and, one-SM shape, into the staging
  // buffers), which the first tile does not use; it stays there until the
  // rows are in TMEM.
  static constexpr uint32_t kOffQ = kOffK + kKBlocks * kKSlotBytes;
  static constexpr uint32_t kQBoxBytes = 64u * kDqk * 2u;   // 64 rows, 72 KB
  static constexpr uint32_t kOffP = 4096;                   // PV: P buffers [kPBufs]
  static constexpr uint32_t kOffV = kOffP + kPBufs * kPBufBytes;        // PV: V ring
  static constexpr uint32_t kEndQK = kOffStage + 2 * kPBufBytes;
  static constexpr uint32_t kEndPV = kOffV + kRingV * kVSlotBytes;
  static constexpr uint32_t kSmemBytes = (kEndQK > kEndPV ? kEndQK : kEndPV) + 1024;

  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(8 * kNumBars <= int(kOffTmemSlot) && kOffFlags + 4 <= kOffValid, "barrier area");
  static_assert(kOffValid + 8 * kValidRing <= kOffPar && kOffPar + 4 * kTmax <= kOffSrow &&
                    kOffMx + 1024 <= kOffK,
                "header");
  static_assert(kOffQ % 1024 == 0 && kOffQ + 2 * kQBoxBytes <= kEndQK, "Q landing area");
  // The Q area starts past tile 0's slots.  Tiles 1 .. kKLag-1 wait for Q to
  // be in TMEM; a later tile waits for a commit of products that came after
  // it, so no copy lands on Q before its rows have left.
};

// Epilogue staging of the PV CTA: 128 rows of 1 KB (512 bf16) + 16 bytes (the
// pad spreads rows over the banks) at kOffP, over the P and value buffers.
constexpr uint32_t kEpiRowBytes = 1024 + 16;
static_assert(4096 + 128 * kEpiRowBytes <= Cfg<false>::kEndPV &&
                  4096 + 128 * kEpiRowBytes <= Cfg<true>::kEndPV,
              "epilogue staging");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemQ = 0;      // QK CTA: Q, 288 columns
constexpr uint32_t kTmemS = 320;    // QK CTA: S buffers at 320 and 384
constexpr long long kWaitCycles = 4000000000ll;   // wait bound in SM cycles (~2 s)
constexpr float kRescaleLog2 = 8.f;
constexpr int kProducers = 224;       // warps 0, 2, 3, 12-15
constexpr uint32_t kProducerBar = 1;  // named barrier of the producer warps
constexpr int kSoftmax = 256;         // warps 4-11
constexpr uint32_t kSoftmaxBar = 2;   // named barrier of the softmax warps

// Products, commits and tensor memory in either shape.  "Local" commits
// arrive on the issuing CTA's barrier (one-SM shape) or on that barrier in
// every CTA of `pair_mask` (the pair); mc commits arrive in `mask` in both.
template <bool kPair>
__device__ __forceinline__ void mma_ts_any(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
  if constexpr (kPair) mma2_ts_warp(d, a, b, idesc, acc);
  else mma_ts_warp(d, a, b, idesc, acc);
}
template <bool kPair>
__device__ __forceinline__ void mma_ss_any(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
  if constexpr (kPair) mma2_ss_warp(d, a, b, idesc, acc);
  else mma_ss_warp(d, a, b, idesc, acc);
}
template <bool kPair>
__device__ __forceinline__ void commit_local(uint32_t bar, uint16_t pair_mask) {
  if constexpr (kPair) mma2_commit_mc_warp(bar, pair_mask);
  else mma_commit_warp(bar);
}
template <bool kPair>
__device__ __forceinline__ void commit_mc(uint32_t bar, uint16_t mask) {
  if constexpr (kPair) mma2_commit_mc_warp(bar, mask);
  else mma_commit_mc_warp(bar, mask);
}

// Two probabilities rounded to bf16 for the PV product; the row sum takes the
// unrounded values so that lse stays exact to fp32 rounding.
__device__ __forceinline__ uint32_t pack_bf16(float a, float b, float& sum) {
  sum += a + b;
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);   // a in the low half
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Raw pool row of key j of the split as stored in the slot list (contiguous
// pools: the row itself; segmented lists: the draft list past the prefix), or
// -1 when j is past the split or the list.  The value is only range-checked
// when it is used, a tile later, so the load's latency overlaps the current
// tile's copies instead of stalling the warp.
__device__ __forceinline__ int fetch_row(const Params& p, const ReqInfo& ri, int j, int k1) {
  if (j >= k1 || j >= ri.nlist) return -1;
  if (p.kv_start) {
    const int64_t r = ri.base + j;
    return (r >= 0 && r < p.num_slots && r <= 0x7fffffff) ? int(r) : -1;
  }
  if (p.draft_slots && j >= ri.P) return __ldg(p.draft_slots + ri.dbase + j);
  return __ldg(p.slot_idx + ri.base + j);
}
// A fetched row, or -1 (no row: the copy zero-fills) when out of the pool.
__device__ __forceinline__ int checked_row(const Params& p, int raw) {
  return (raw >= 0 && int64_t(raw) < p.num_slots) ? raw : -1;
}

// Producer warps (224 threads): bring the CTA's share of each 64-key tile
// into its ring slots in the 128B-swizzled K-major layout (block j of the
// share -> slot (nb*t + j) mod kRing; inside a slot row `key`, 16-byte chunk
// (c%8) ^ (key%8)).  The share: every key and column block, or in a pair the
// CTA's half of the keys (QK: keys 32h .. 32h+31, all nine blocks) or of the
// value blocks (PV: blocks {0,1,4,5} + 2h), h = the CTA's rank in the pair.
//  - Paged keys, or a split's ragged last tile: 16-byte cp.async copies, one
//    warp per key (lane l copies chunks l, l+32, l+64 of the share, so one
//    warp instruction moves up to 512 bytes of the row), zero-filled for keys
//    without a row.  The tile's 64 pool rows are staged in shared memory and
//    fetched one tile ahead.
//  - Contiguous keys (kv_start) for a whole in-range tile: TMA tiled box
//    loads.  When the tile's slots do not wrap around the ring, one 3-D box
//    (64 columns x keys x column blocks, map `map3`) lands the share (a PV
//    pair CTA: two boxes of two blocks); otherwise one box per column block
//    (2-D map `map2`).
// Before filling a tile, producer 0 waits for the release of its slots by the
// products of the tiles that used them before (value side: the slot of the
// tile's last block; key side: one commit per tile, see Cfg).  With kMask the
// tile's 64-bit key-validity mask (all 64 keys) goes to the ring read by the
// softmax warps.  Completion: every producer's cp.async arrival (noinc) on the
// tile's full barrier plus one arrival of producer 0 (carrying the TMA byte
// count when boxes are used).  Returns false when a bounded wait gave up (all
// producers agree through the named barrier).  Keys without a valid pool row
// set VA_STATUS_BAD_SLOT in the CTA's status word `cta_flags` (shared memory).
#ifdef VA_TEST_HOOKS
// Bounded wait for a device flag to become non-zero (test gate).
__device__ __noinline__ bool gate_wait(const int32_t* flag, long long limit_cycles) {
  const long long t0 = clock64();
  while (*reinterpret_cast<const volatile int32_t*>(flag) == 0) {
    if (clock64() - t0 > limit_cycles) return false;
    __nanosleep(2000);
  }
  return true;
}
#endif

template <bool kPair, int kBlocks, int kRing, bool kMask>
__device__ __forceinline__ bool produce(const Params& p, const ReqInfo& ri, const SplitRange& sr,
                                        int ntiles, int ptid, uint32_t ring, uint32_t full0,
                                        uint32_t empty0, int* srow, uint32_t* valid32,
                                        uint32_t vready0, volatile int* abort_flag,
                                        const CUtensorMap* map3, const CUtensorMap* map2,
                                        bool box3d, uint32_t qready, int raw,
                                        uint32_t* cta_flags, int hh) {
  using C = Cfg<kPair>;
  constexpr int kKeys = kMask ? C::kSlotKeys : kTile;      // keys of the share per tile
  constexpr uint32_t kSlot = uint32_t(kKeys) * 128u;       // slot bytes
  constexpr int kChunks = kBlocks * 8;                     // 16-byte chunks of a key's share
  const int koff = kMask ? hh * kKeys : 0;                 // first key of the share
  // pool column block of the share's block j
  auto col_block = [&](int j) -> int {
    return (kPair && !kMask) ? (j & 1) + 4 * (j >> 1) + 2 * hh : j;
  };
  const int lane = ptid & 31;
  bool ok = true;
  bool bad_slot = false;
#ifdef VA_TEST_HOOKS
  {
    bool open = true;
    if (ptid == 0 && g_va_test_gate) open = gate_wait(g_va_test_gate, kWaitCycles);
    if (!named_sync_and(kProducerBar, kProducers, open)) return false;
  }
#endif
  // the last box-loaded tile at each full barrier (-1: none, or a tile of
  // copies since), drained below if a wait gives up while they are in flight
  int box_tile[C::kFullRing];
#pragma unroll
  for (int i = 0; i < C::kFullRing; ++i) box_tile[i] = -1;
  VA_PH_DECL;
  for (int t = 0; t < ntiles; ++t) {
    const int g0 = kBlocks * t;   // ring position of the tile's first block
    const int s0 = g0 % kRing;
    bool got = true;
    // Producer 0 waits for the release of the tile's slots once.  (One
    // blocking wait per tile: each one costs a wake-up latency, and nine in a
    // row cost more than the deeper ring gains.)  The others learn the
    // outcome at the named barrier below.
    if (kMask) {
      // QK side: one commit per tile covers every earlier product (a commit
      // arrives only once all earlier products have completed); each commit
      // costs the issuing warp about as much as an N=64 product, so the QK
      // products commit twice per tile, not once per slot.  Tiles 1 ..
      // kKLag-1 hold Q until its rows are in TMEM.
      if (ptid == 0 && t >= C::kKLag) {
        const int u = t - C::kKLag;
        got = mbar_wait(empty0 + 8u * uint32_t(u % C::kKEmptyRing),
                        uint32_t(u / C::kKEmptyRing) & 1u, abort_flag, kWaitCycles);
      }
      if (ptid == 0 && t >= 1 && t < C::kKLag) got = mbar_wait(qready, 0, abort_flag, kWaitCycles);
    } else {
      // value side: the slot of the tile's last block; its previous occupant
      // is the latest of the previous occupants in issue order
      const int g = g0 + kBlocks - 1;
      if (ptid == 0 && g >= kRing)
        got = mbar_wait(empty0 + 8u * uint32_t(g % kRing), uint32_t(g / kRing - 1) & 1u, abort_flag,
                        kWaitCycles);
    }
    if (ptid == 0) VA_TRACE_EVENT(kMask ? 0 : 3, 0, t);
    VA_PH(0);
    if (ptid < 64) {
      const int rw = checked_row(p, raw);
      srow[(t & 1) * 64 + ptid] = rw;
      if (kMask) {
        const int j = sr.k0 + t * kTile + ptid;
        bad_slot |= j < sr.k1 && rw < 0;
        const uint32_t bal = __ballot_sync(0xffffffffu, rw >= 0);
        if (lane == 0) valid32[(t % C::kValidRing) * 2 + (ptid >> 5)] = bal;
      }
    }
    if (!named_sync_and(kProducerBar, kProducers, got)) {
      ok = false;
      break;
    }
    VA_PH(1);
    const int fi = t % C::kFullRing;
    const uint32_t fb = full0 + 8u * uint32_t(fi);
    // contiguous rows, whole tile inside the split and the pool: box loads
    const int tk0 = sr.k0 + t * kTile;
    // a tile with draft keys, when the call appends their rows first: after
    // the append (in the kernel before this one) has completed
    if (p.draft_kv && tk0 + kTile > ri.P) griddep_wait();
    const int64_t row0 = p.kv_start ? ri.base + tk0 : -1;
    bool boxes = p.kv_start != nullptr && tk0 + kTile <= sr.k1 && tk0 + kTile <= ri.nlist &&
                 row0 >= 0 && row0 + kTile <= p.num_slots && row0 + kTile <= 0x7fffffff;
    if (kPair && !kMask && !box3d) boxes = false;   // the PV pair share needs the 3-D map
    if (kMask && ptid == 0) mbar_arrive(vready0 + 8u * uint32_t(t % C::kValidRing));
    if (ptid == 0) {
      box_tile[fi] = boxes ? t : -1;
      if (boxes) {
        mbar_arrive_expect_tx(fb, uint32_t(kBlocks) * kSlot);
        if (kPair && !kMask) {
          // blocks {0,1} + 2h and {4,5} + 2h: adjacent slot pairs (a value
          // tile never wraps: the ring is a multiple of 4 slots)
          tma_load_3d(ring + uint32_t(s0) * kSlot, map3, 0, int(row0), 2 * hh, fb);
          tma_load_3d(ring + uint32_t(s0 + 2) * kSlot, map3, 0, int(row0), 4 + 2 * hh, fb);
        } else if (box3d && s0 + kBlocks <= kRing) {
          tma_load_3d(ring + uint32_t(s0) * kSlot, map3, 0, int(row0) + koff, 0, fb);
        } else {
#pragma unroll 1
          for (int c = 0; c < kBlocks; ++c) {
            const int sl = s0 + c < kRing ? s0 + c : s0 + c - kRing;
            tma_load_2d(ring + uint32_t(sl) * kSlot, map2, 64 * c, int(row0) + koff, fb);
          }
        }
      } else {
        mbar_arrive(fb);
      }
    }
    if (ptid < 64 && t + 1 < ntiles) raw = fetch_row(p, ri, sr.k0 + (t + 1) * kTile + ptid, sr.k1);
    if (!boxes) {
      // this lane's chunks lane + 32j lie in the share's blocks lane/8 + 4j,
      // at chunk position lane%8 inside their 128-byte row
      uint32_t slot_addr[3];
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int cb = (lane >> 3) + 4 * j;
        const int sl = s0 + cb < kRing ? s0 + cb : s0 + cb - kRing;
        slot_addr[j] = ring + uint32_t(sl) * kSlot;
      }
      const int pw = ptid >> 5;
      // a PV pair CTA's single chunk per key (its four blocks, 32 chunks):
      // pool column of the lane's chunk
      const int vcol = col_block(lane >> 3) * 64 + (lane & 7) * 8;
#pragma unroll 2
      for (int key = pw; key < kKeys; key += kProducers / 32) {
        const int row = srow[(t & 1) * 64 + koff + key];
        const __nv_bfloat16* src = p.kv + (row >= 0 ? int64_t(row) * p.kv_stride : 0);
        const uint32_t nb = row >= 0 ? 16u : 0u;
        const uint32_t kx = uint32_t(key) * 128u + uint32_t(((lane & 7) ^ (key & 7)) * 16);
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int c = lane + 32 * j;
          if (c < kChunks) {
            // (the plain c * 8 keeps the one-SM gather's address arithmetic
            // minimal: a general block map here cost 3 % on paged pools)
            if constexpr (kPair && !kMask) cp_async16(slot_addr[j] + kx, src + vcol, nb);
            else cp_async16(slot_addr[j] + kx, src + c * 8, nb);
          }
        }
      }
    }
    cp_async_arrive_noinc(fb);
    if (ptid == 0) VA_TRACE_EVENT(kMask ? 0 : 3, 1, t);
    VA_PH(2);
  }
  if (ptid == 0) VA_PH_STORE((kMask ? 11 : 12) + 3 * hh);
  cp_async_wait_all();
  // After a wait gave up, the boxes still in flight land before the CTA can
  // leave.  Each full barrier's last issued tile received all of its
  // arrivals, and no later phase of that barrier can complete, so the parity
  // wait is exact; boxes of earlier tiles at that barrier had landed before
  // it was reused.
  if (!ok && ptid == 0)
    for (int i = 0; i < C::kFullRing; ++i)
      if (box_tile[i] >= 0)
        (void)mbar_wait(full0 + 8u * uint32_t(i), uint32_t(box_tile[i] / C::kFullRing) & 1u,
                        nullptr, kWaitCycles);
  if (kMask && bad_slot) atomicOr(cta_flags, VA_STATUS_BAD_SLOT);
  return ok;
}

// Q rows into TMEM as the A operand (bf16 pairs, 288 columns), from the
// shared landing area that the row block's two TMA boxes filled.  The two
// softmax warpgroups share the work: warp w writes lane quadrant w%4 (rows
// 32*(w%4) .. +31) for column blocks 0-4 (first warpgroup) or 5-8 (second).
// Lane r reads its row's 128-byte piece of a column block as eight 16-byte
// chunks (chunk j sits at position j ^ (r%8) of the swizzled row) and stores
// it with one tcgen05.st.  Returns false when the bounded wait for the boxes
// gave up.
__device__ __forceinline__ bool load_q(int half, int q4, int lane, uint32_t tmem, uint32_t qs,
                                       uint32_t qbar, volatile int* abort_flag) {
  constexpr uint32_t kQBoxBytes = Cfg<false>::kQBoxBytes;
  constexpr uint32_t kQBlockBytes = 64u * 128u;   // one column block of a 64-row box
  const bool ok = mbar_wait(qbar, 0, abort_flag, kWaitCycles);
  const int c_begin = half ? 5 : 0, c_end = half ? 9 : 5;
  const uint32_t tl = tmem + (uint32_t(q4 * 32) << 16) + kTmemQ;
  const int r = q4 * 32 + lane;   // row of the block
  const uint32_t row_addr = qs + uint32_t(r >> 6) * kQBoxBytes + uint32_t(r & 63) * 128u;
  if (ok) {
#pragma unroll 1
    for (int c = c_begin; c < c_end; ++c) {
      uint32_t v[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 w = ld_shared_v4(row_addr + uint32_t(c) * kQBlockBytes + uint32_t((j ^ (r & 7)) * 16));
        v[4 * j] = w.x; v[4 * j + 1] = w.y; v[4 * j + 2] = w.z; v[4 * j + 3] = w.w;
      }
      tmem_st32(tl + 32u * uint32_t(c), v);
    }
  }
  tmem_wait_st();
  return ok;
}

template <bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    partial_tc_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v,
                      const __grid_constant__ CUtensorMap tmap_2d,
                      const __grid_constant__ CUtensorMap tmap_q, int box3d) {
  using C = Cfg<kPair>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sb - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + C::kOffAbort);
  auto bar = [&](int i) -> uint32_t { return sb + C::kOffBars + 8u * uint32_t(i); };

  const uint32_t rank = cluster_ctarank();
  // Role (QK or PV) and rows: hh = which 128 rows of the unit (a pair's
  // ranks); `other` = the CTA of the other role for the same rows; `mate` =
  // the other CTA of a pair (the even one issues both CTAs' products).
  const bool qk = kPair ? rank < 2u : rank == 0u;
  const int hh = kPair ? int(rank & 1u) : 0;
  const bool issuer_cta = hh == 0;
  const uint32_t other = kPair ? (rank ^ 2u) : (rank ^ 1u);
  const uint32_t mate = rank ^ 1u;
  const int split = blockIdx.x / C::kCtas, rb = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#ifdef VA_TRACE
  const int trace_role = rank < 2u ? 6 + int(rank) : 14 + int(rank);   // per-CTA marks
#endif
  if (tid == 0) VA_TRACE_CTA(trace_role, 0);
  // the maps' descriptors are fetched while the request's bounds load
  if (tid == 0) {
    if (qk) tma_prefetch(&tmap_q);
    if (p.kv_start) {
      tma_prefetch(qk ? &tmap_k : &tmap_v);
      tma_prefetch(&tmap_2d);
    }
  }

  // The kernel computes its rows' ancestor masks itself and keeps its status
  // bits in shared memory, stored to its own workspace word at the end; the
  // merge kernel ORs those into the status word.  It is the call's first
  // kernel, launched as a programmatic dependent of the stream's previous
  // kernel: its clusters may be resident while that kernel finishes, and
  // wait here, before reading any input, until it has completed.  When the
  // call appends draft rows first, the append kernel (launched after the
  // stream's earlier work) precedes it instead, and the producers wait
  // (griddepcontrol.wait) only before a tile holding draft keys.
  if (!p.draft_kv) griddep_wait();
  // the merge kernel may be scheduled as clusters retire (only after the
  // wait above: it reads the call's bounds before its own wait)
  griddep_launch_dependents();
  const ReqInfo ri = req_info(p, b, false);
  const SplitRange sr = split_range(ri.N, p.nsplit, split);
  // this CTA's status word, for the merge kernel to OR into the status word
  // (words [request][128-row block][split][QK, PV]; every CTA of the grid
  // owns one and stores it, so the merge ORs them all without bounds)
  uint32_t* const flag_word =
      p.cta_flags +
      ((size_t(b) * p.flag_blocks + (kPair ? 2 * rb + hh : rb)) * p.nsplit + split) * 2 + (qk ? 0 : 1);
  if (split >= sr.nsplit_eff) {   // every CTA of the cluster leaves together
    if (threadIdx.x == 0) *flag_word = 0u;
    return;
  }
  const int R = p.rows_per_req;
  const int row0 = rb * C::kUnitRows + hh * kRows;
  const int ntiles = ceil_div(sr.k1 - sr.k0, kTile);
  const size_t rows_total = size_t(p.B) * R;

  const bool producer = warp == 0 || warp == 2 || warp == 3 || warp >= 12;
  const int ptid = warp == 0 ? lane : (warp < 4 ? warp - 1 : warp - 9) * 32 + lane;
  // raw pool rows of the first tile (producers), loaded during the set-up
  const int raw0 = producer && ptid < 64 ? fetch_row(p, ri, sr.k0 + ptid, sr.k1) : -1;

  uint32_t* cta_flags = reinterpret_cast<uint32_t*>(gb + C::kOffFlags);
  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(cta_flags, VA_STATUS_TIMEOUT);
  };

  if (tid == 0) {
    for (int i = 0; i < C::kNumBars; ++i) {
      uint32_t cnt = 1;
      // in a pair the odd rank's eight softmax (row) warps add one arrival each
      if (i == C::B_SEMPTY || i == C::B_SEMPTY + 1 || i == C::B_OCORR)
        cnt = kSoftmax + (kPair ? kSoftmax / 32 : 0);
      if (i == C::B_QREADY) cnt = kSoftmax;
      if (kPair && i == C::B_QREADYP) cnt = kSoftmax / 32;
      if (i >= C::B_FULL && i < C::B_FULL + C::kFullRing) cnt = kProducers + 1;   // copies + producer 0
      if (i == C::B_FIN) cnt = 4;   // one per warp of the first softmax warpgroup
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    *cta_flags = 0u;
    fence_mbar_init();
  }
  if (warp == 2) {
    if constexpr (kPair) tmem_alloc_pair(sb + C::kOffTmemSlot, kTmemCols);
    else tmem_alloc(sb + C::kOffTmemSlot, kTmemCols);
  }
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gb + C::kOffTmemSlot);
  if (tid == 0) VA_TRACE_CTA(trace_role, 1);
  int* srow = reinterpret_cast<int*>(gb + C::kOffSrow);
  const int half = (warp - 4) >> 2;   // softmax / row warpgroup (warps >= 4)
  const int q4 = warp & 3;            // TMEM lane quadrant of the warp

  if (qk) {
    // ================================================================ QK CTA
    volatile uint64_t* valid_ring = reinterpret_cast<volatile uint64_t*>(gb + C::kOffValid);
    if (producer) {
      // ---- producers: the CTA's keys of each tile (all 576 columns)
      if (!produce<kPair, kKBlocks, C::kRingK, true>(
              p, ri, sr, ntiles, ptid, sb + C::kOffK, bar(C::B_FULL), bar(C::B_EMPTY), srow,
              reinterpret_cast<uint32_t*>(gb + C::kOffValid), bar(C::B_VREADY), abort_flag,
              &tmap_k, &tmap_2d, box3d != 0, bar(C::B_QREADY), raw0, cta_flags, hh) &&
          ptid == 0)
        fail();
    } else if (warp == 1) {
      // The row block's Q: two boxes of 64 rows x 9 column blocks (rows past
      // the tensor read as zeros; rows of the next request are never used).
      // Issued here, after the cluster barrier: issued before it, the copy
      // in flight held the barrier back by about half a microsecond.
      if (lane == 0) {
        const int qrow = b * R + row0;
        mbar_arrive_expect_tx(bar(C::B_QTMA), 2u * C::kQBoxBytes);
        tma_load_3d(sb + C::kOffQ, &tmap_q, 0, qrow, 0, bar(C::B_QTMA));
        tma_load_3d(sb + C::kOffQ + C::kQBoxBytes, &tmap_q, 0, qrow + 64, 0, bar(C::B_QTMA));
      }
      __syncwarp();
      if (issuer_cta) {
        // ---- MMA issuer: S[t%2] = Q K_t^T.  The whole warp runs the loop
        // and one elected lane issues, 36 MMAs back to back with fixed
        // descriptor offsets, so the tensor pipe sees them at its own rate.
        bool ok = __all_sync(0xffffffffu,
                             mbar_wait(bar(C::B_QREADY), 0, abort_flag, kWaitCycles) &&
                                 (!kPair || mbar_wait<true>(bar(C::B_QREADYP), 0, abort_flag,
                                                            kWaitCycles)));
        if (!ok && lane == 0) fail();
        constexpr uint32_t idesc = idesc_bf16(C::kUnitRows, 64, 0, 0);
        VA_PH_DECL;
        for (int t = 0; ok && t < ntiles; ++t) {
          const int bs = t & 1;
          const int fi = t % C::kFullRing;
          const uint32_t fpar = uint32_t(t / C::kFullRing) & 1u;
          const bool got =
              mbar_wait(bar(C::B_FULL + fi), fpar, abort_flag, kWaitCycles) &&
              (!kPair || mbar_wait<true>(bar(C::B_FULLP + fi), fpar, abort_flag, kWaitCycles)) &&
              (t < 2 || mbar_wait<kPair>(bar(C::B_SEMPTY + bs), uint32_t((t >> 1) - 1) & 1u,
                                         abort_flag, kWaitCycles));
          VA_PH(0);
          if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) fail();
            break;
          }
          fence_proxy_async_cta();   // the producers' cp.async writes, seen by the tensor core
          tc_fence_after();
          if (lane == 0) VA_TRACE_EVENT(1, 0, t);
          const int s0 = (kKBlocks * t) % C::kRingK;
          const uint32_t d = tmem + kTmemS + 64u * uint32_t(bs);
          // K columns 16k..16k+15 (k = 4c + kk): column block c in its ring
          // slot, 32-byte step kk inside the swizzled row (the descriptor's
          // address field counts 16-byte units).  Two commits per tile:
          // blocks 0..kKRelease read (the producers refill those slots kKLag
          // tiles on), then the whole tile (S ready, every slot read).  A
          // commit costs an N=64 product's issue slot (measured: 45 cycles per
          // product with a commit after every fourth, 34.5 without), so the
          // slots are not released one by one.
#pragma unroll
          for (int c = 0; c < kKBlocks; ++c) {
            const int sl = s0 + c < C::kRingK ? s0 + c : s0 + c - C::kRingK;
            const uint64_t bd = smem_desc(sb + C::kOffK + uint32_t(sl) * C::kKSlotBytes, 16, 1024,
                                          kSwizzle128B);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts_any<kPair>(d, tmem + kTmemQ + 8u * uint32_t(4 * c + kk),
                                bd + uint64_t((uint32_t(kk) * 32u) >> 4), idesc,
                                (c | kk) != 0 ? 1u : 0u);
            if (c == C::kKRelease)
              commit_local<kPair>(bar(C::B_EMPTY + t % C::kKEmptyRing), C::kQkMask);
          }
          commit_local<kPair>(bar(C::B_SFULL + bs), C::kQkMask);
          if (lane == 0) VA_TRACE_EVENT(1, 1, t);
          VA_PH(2);
        }
        if (lane == 0) VA_PH_STORE(9);
        commit_local<kPair>(bar(C::B_MMAFIN), C::kQkMask);
        mbar_wait(bar(C::B_MMAFIN), 0, nullptr, kWaitCycles);
      } else {
        // ---- odd rank of the QK pair: forwards each key tile's arrival to
        // the even rank, whose products read this CTA's slots
        const uint32_t fullp = mapa(bar(C::B_FULLP), mate);
        for (int t = 0; t < ntiles; ++t) {
          const int fi = t % C::kFullRing;
          if (!__all_sync(0xffffffffu, mbar_wait(bar(C::B_FULL + fi), uint32_t(t / C::kFullRing) & 1u,
                                                 abort_flag, kWaitCycles))) {
            if (lane == 0) fail();
            break;
          }
          fence_proxy_async_cta();   // this CTA's cp.async writes, read by the pair's tensor core
          if (lane == 0) mbar_arrive_remote(fullp + 8u * uint32_t(fi));
          __syncwarp();
        }
        // the even rank's products read this CTA's shared memory and write its
        // tensor memory until their last commit
        (void)mbar_wait(bar(C::B_MMAFIN), 0, nullptr, kWaitCycles);
      }
      // the Q boxes this lane issued have landed before the CTA can leave
      // (normally long since; after an abort, possibly not)
      if (lane == 0) (void)mbar_wait(bar(C::B_QTMA), 0, nullptr, kWaitCycles);
      __syncwarp();
    } else if (warp >= 4) {
      // ---- softmax: warpgroup `half` owns columns [32*half, 32*half + 32) of
      // every tile for row r
      // the request's tree parents, staged for the ancestor walk below while
      // Q is on its way
      int* par = reinterpret_cast<int*>(gb + C::kOffPar);
      if (p.tree_parent && tid - 128 < p.T) par[tid - 128] = p.tree_parent[size_t(b) * p.T + (tid - 128)];
      if (!load_q(half, q4, lane, tmem, sb + C::kOffQ, bar(C::B_QTMA), abort_flag) && tid == 128)
        fail();
      tc_fence_before();
      mbar_arrive(bar(C::B_QREADY));
      if (kPair && !issuer_cta) {
        // the even rank's products read this CTA's Q rows too
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa(bar(C::B_QREADYP), mate));
      }
      if (split == 0 && rb == 0 && hh == 0 && tid == 128) {
        bool bad = false;
        (void)req_info(p, b, false, &bad);
        if (bad) atomicOr(cta_flags, VA_STATUS_BAD_INDPTR);
      }
      if (tid == 128) VA_TRACE_CTA(6, 5);
      const int r = q4 * 32 + lane;
      const int lr = row0 + r;
      const bool row_ok = lr < R;
      const bool issuer = warp == 4 && lane == 0;
      const uint32_t tl = tmem + (uint32_t(q4 * 32) << 16);
      // The row's draft node and its ancestor-or-self set (bit k: draft node
      // k), from the parents (a walk up the staged list: a node whose parent
      // is not an earlier node hangs off the prefix and is flagged, and a walk
      // stops below such a node), from the dense mask rows (the last T
      // entries of the node's row; entries past the mask read as 0 and are
      // flagged), or as the caller gave them.
      named_sync(kSoftmaxBar, kSoftmax);   // parents staged
      uint64_t nbits = 0ull;
      if (row_ok) {
        const int node = lr / p.H;
        if (p.tree_parent) {
          nbits = 1ull << node;
          int q = par[node];
          if (q < -1 || q >= node) {
            atomicOr(cta_flags, VA_STATUS_BAD_PARENT);
          } else {
            while (q >= 0) {
              nbits |= 1ull << q;
              const int up = par[q];
              if (up < -1 || up >= q) break;
              q = up;
            }
          }
        } else if (p.dense_mask) {
          const int64_t first = p.kv_indptr[0];
          const int64_t e0 = int64_t(p.T) * ((ri.base - first) + int64_t(b) * p.T) +
                             int64_t(node) * (ri.P + p.T) + ri.P;
          bool bad = false;
          for (int k = 0; k < p.T; ++k) {
            const int64_t e = e0 + k;
            if (e >= 0 && e < p.dense_mask_len) {
              if (p.dense_mask[e]) nbits |= 1ull << k;
            } else {
              bad = true;
            }
          }
          if (bad) atomicOr(cta_flags, VA_STATUS_BAD_MASK);
        } else {
          nbits = p.bits[size_t(b) * p.T + node];
        }
      }
      float* mx = reinterpret_cast<float*>(gb + C::kOffMx);
      const uint32_t pv_p = mapa(sb + C::kOffP, other);
      const uint32_t pv_pfull = mapa(bar(C::B_PFULL), other);
      const uint32_t pv_fin = mapa(sb + C::kOffFin, other);
      const uint32_t pv_finbar = mapa(bar(C::B_FIN), other);
      const uint32_t sempty_issuer = kPair ? mapa(bar(C::B_SEMPTY), mate) : 0u;
      float m_ref = -INFINITY, l = 0.f;
      bool issuer_ok = true;
      bool ok = true;
      VA_PH_DECL;
      for (int t = 0; t < ntiles; ++t) {
        const int bs = t & 1;             // S buffer and staging buffer
        const int pb = t % kPBufs;        // P buffer of the PV CTA
        const int tk0 = sr.k0 + t * kTile;
        // visibility: prefix keys always, draft key k when bit k of the node's mask
        const int off = ri.P - tk0;
        uint64_t vis;
        if (off >= 64) {
          vis = ~0ull;
        } else if (off > 0) {
          vis = ((1ull << off) - 1ull) | (nbits << off);
        } else {
          vis = (-off) >= 64 ? 0ull : (nbits >> (-off));
        }
        if (!row_ok) vis = 0ull;

        // S_t ready, and the producers' validity mask of this tile
        const bool got =
            mbar_wait(bar(C::B_SFULL + bs), uint32_t(t >> 1) & 1u, abort_flag, kWaitCycles) &&
            mbar_wait(bar(C::B_VREADY + t % C::kValidRing), uint32_t(t / C::kValidRing) & 1u,
                      abort_flag, kWaitCycles);
        VA_PH(0);
        const bool wok = __all_sync(0xffffffffu, got);
        float x[32];
        float mth = -INFINITY;
        if (wok) {
          const uint32_t v32 =
              uint32_t(((vis & valid_ring[t % C::kValidRing]) >> (32 * half)));
          if (tid == 128) VA_TRACE_EVENT(2, 0, t);
          tc_fence_after();
          uint32_t sv[32];
          tmem_ld32(tl + kTmemS + 64u * uint32_t(bs) + 32u * uint32_t(half), sv);
          tmem_wait_ld();
          tc_fence_before();
          if (!kPair || issuer_cta) {
            mbar_arrive(bar(C::B_SEMPTY + bs));
          } else {
            // the warp's S loads have completed (wait::ld above): a relaxed
            // arrival suffices, and a cluster-scope release here cost about
            // 1100 cycles per tile on the softmax chain
            __syncwarp();
            if (lane == 0) mbar_arrive_remote_relaxed(sempty_issuer + 8u * uint32_t(bs));
          }
          // With a positive scale (the usual case) the raw scores are kept
          // (hidden keys -inf), their maximum is scaled once, and each
          // exponent below is one fused multiply-add (x * scale - m); a tile
          // whose keys are all visible skips the mask.  Otherwise the scores
          // are scaled here and the multiply-add's factor is 1.
          if (p.scale_log2 > 0.f) {
            if (v32 == 0xffffffffu) {
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                x[c] = __uint_as_float(sv[c]);
                mth = fmaxf(mth, x[c]);
              }
            } else {
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                x[c] = ((v32 >> c) & 1u) ? __uint_as_float(sv[c]) : -INFINITY;
                mth = fmaxf(mth, x[c]);
              }
            }
            mth *= p.scale_log2;
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              x[c] = ((v32 >> c) & 1u) ? __uint_as_float(sv[c]) * p.scale_log2 : -INFINITY;
              mth = fmaxf(mth, x[c]);
            }
          }
        }
        VA_PH(1);
        mx[half * kRows + r] = mth;
        if (issuer) bulk_wait_read<1>();   // staging buffer bs: tile t-2's copy has read it
        if (!named_sync_and(kSoftmaxBar, kSoftmax, wok && issuer_ok)) {
          if (issuer) fail();
          ok = false;
          break;
        }
        VA_PH(2);
        const float mt = fmaxf(mx[r], mx[kRows + r]);
        float alpha = 1.f;
        if (mt > m_ref + kRescaleLog2) {
          alpha = ex2_approx(m_ref - mt);   // 0 when nothing was seen before
          l *= alpha;
          m_ref = mt;
        }
        const float mr = m_ref == -INFINITY ? 0.f : m_ref;
        const float sc = p.scale_log2 > 0.f ? p.scale_log2 : 1.f;
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = pack_bf16(ex2_approx(fmaf(x[2 * c], sc, -mr)),
                            ex2_approx(fmaf(x[2 * c + 1], sc, -mr)), l);
        if (tid == 128) VA_TRACE_EVENT(2, 1, t);
        VA_PH(3);
        // this row's 32 keys into the staging buffer (K-major, 128B swizzle)
        uint8_t* stg = gb + C::kOffStage + uint32_t(bs) * kPBufBytes;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int chunk = 4 * half + j;
          *reinterpret_cast<uint4*>(stg + r * 128 + ((chunk ^ (r & 7)) * 16)) =
              make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
        if (half == 0) {
          reinterpret_cast<float*>(stg + kPAlpha)[r] = alpha;
          const uint32_t wres = __ballot_sync(0xffffffffu, alpha != 1.f);
          if (lane == 0)
            reinterpret_cast<uint32_t*>(stg + kPFlags)[q4] = (uint32_t(t) << 1) | (wres ? 1u : 0u);
        }
        fence_proxy_async_cta();   // staging writes, read by the bulk copy
        VA_PH(4);
        named_sync(kSoftmaxBar, kSoftmax);
        VA_PH(5);
        if (issuer) {
          issuer_ok = t < kPBufs ||
                      mbar_wait<true>(bar(C::B_PFREE + pb), uint32_t((t / kPBufs) - 1) & 1u,
                                      abort_flag, kWaitCycles);
          if (tid == 128) VA_TRACE_EVENT(2, 2, t);
          if (issuer_ok) {
            // the PV CTA armed this buffer's barrier with the byte count
            bulk_copy_to_cluster(pv_p + uint32_t(pb) * kPBufBytes, smem_u32(stg), kPPayload,
                                 pv_pfull + 8u * uint32_t(pb));
            bulk_commit();
          }
          if (tid == 128) VA_TRACE_EVENT(2, 3, t);
        }
        VA_PH(6);
      }
      if (tid == 128) VA_PH_STORE(8 + 5 * hh);
      // row sums: the two warpgroups' partial sums share the reference max
      if (ok) {
        mx[half * kRows + r] = l;
        named_sync(kSoftmaxBar, kSoftmax);
        if (half == 0) {
          const float lt = mx[r] + mx[kRows + r];
          const float lse = lt > 0.f ? (m_ref + log2f(lt)) * kLn2 : -INFINITY;
          if (row_ok) p.part_lse[size_t(split) * rows_total + size_t(b) * R + lr] = lse;
          st_cluster_f32(pv_fin + uint32_t(r) * 4u, lt > 0.f ? 1.f / lt : 0.f);
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(pv_finbar);
        }
      }
      if (issuer) {
        // the last copies have read the staging buffers, and the PV CTA's last
        // releases of the P buffers have landed, before shared memory goes away
        bulk_wait_read<0>();
        if (ok)
          for (int t = ntiles - kPBufs > 0 ? ntiles - kPBufs : 0; t < ntiles; ++t)
            if (!mbar_wait<true>(bar(C::B_PFREE + t % kPBufs), uint32_t(t / kPBufs) & 1u,
                                 abort_flag, kWaitCycles))
              fail();
      }
    }
  } else {
    // ================================================================ PV CTA
    volatile uint32_t* cmd = reinterpret_cast<volatile uint32_t*>(gb + C::kOffCmd);
    if (producer) {
      // ---- producers: the CTA's value columns of the same tiles
      if (!produce<kPair, C::kVBlocksCta, kRingV, false>(
              p, ri, sr, ntiles, ptid, sb + C::kOffV, bar(C::B_FULL), bar(C::B_EMPTY), srow,
              nullptr, 0u, abort_flag, &tmap_v, &tmap_2d, box3d != 0, 0u, raw0, cta_flags, hh) &&
          ptid == 0)
        fail();
      if constexpr (!kPair) cluster_arrive_relaxed();   // done with the QK CTA (see the end)
    } else if (warp == 1 && issuer_cta) {
      // ---- MMA issuer: O += P_t V_t (whole warp, one elected lane issues)
      constexpr uint32_t idesc = idesc_bf16(C::kUnitRows, 256, 0, 1);
      uint32_t nresc = 0;
      // a pair's odd rank: its command word and rescale barrier
      const uint32_t m_cmd = kPair ? mapa(sb + C::kOffCmd, mate) : 0u;
      const uint32_t m_ogo = kPair ? mapa(bar(C::B_OGO), mate) : 0u;
      // each P buffer's barrier expects one arrival (ours, carrying the byte
      // count of the QK CTA's bulk copy into it): arm the first uses now
      if (lane == 0)
        for (int t = 0; t < kPBufs && t < ntiles; ++t)
          mbar_arrive_expect_tx(bar(C::B_PFULL + t), kPPayload);
      __syncwarp();
      VA_PH_DECL;
      for (int t = 0; t < ntiles; ++t) {
        const int bs = t % kPBufs;
        const int fi = t % C::kFullRing;
        const uint32_t fpar = uint32_t(t / C::kFullRing) & 1u;
        const uint32_t ppar = uint32_t(t / kPBufs) & 1u;
        const bool got =
            mbar_wait(bar(C::B_FULL + fi), fpar, abort_flag, kWaitCycles) &&
            mbar_wait<true>(bar(C::B_PFULL + bs), ppar, abort_flag, kWaitCycles) &&
            (!kPair || mbar_wait<true>(bar(C::B_FULLP + fi), fpar, abort_flag, kWaitCycles));
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) fail();
          break;
        }
        if (lane == 0) VA_TRACE_EVENT(4, 0, t);
        VA_PH(0);
        const uint32_t pbase = sb + C::kOffP + uint32_t(bs) * kPBufBytes;
        const volatile uint32_t* flags =
            reinterpret_cast<const volatile uint32_t*>(gb + C::kOffP + bs * kPBufBytes + kPFlags);
        uint32_t any = 0;
#pragma unroll
        for (int w = 0; w < 4; ++w) any |= flags[w] & 1u;
        // the odd rank's rows: its forwarder stored their flag before arriving
        if constexpr (kPair)
          any |= reinterpret_cast<const volatile uint32_t*>(gb + C::kOffPeerAny)[bs];
        if (__any_sync(0xffffffffu, any != 0) && t > 0) {
          // rows change reference: O must be final for tile t-1 before the
          // row warps rescale it, and rescaled before this tile's product
          commit_local<kPair>(bar(C::B_ODONE), uint16_t(1u << rank));
          bool g = __all_sync(0xffffffffu,
                              mbar_wait(bar(C::B_ODONE), nresc & 1u, abort_flag, kWaitCycles));
          if (g) {
            if (lane == 0) {
              *cmd = uint32_t(bs);
              mbar_arrive(bar(C::B_OGO));
              if constexpr (kPair) {
                st_cluster_u32(m_cmd, uint32_t(bs));
                mbar_arrive_remote(m_ogo);
              }
            }
            __syncwarp();
            g = __all_sync(0xffffffffu,
                           mbar_wait<kPair>(bar(C::B_OCORR), nresc & 1u, abort_flag, kWaitCycles));
          }
          ++nresc;
          if (!g) {
            if (lane == 0) fail();
            break;
          }
        }
        VA_PH(1);
        fence_proxy_async_cta();
        tc_fence_after();
        const uint64_t ad0 = smem_desc(pbase, 16, 1024, kSwizzle128B);
        const int s0 = (C::kVBlocksCta * t) % kRingV;
        // O columns [256q, 256q+256) += P keys 16k..16k+15 x V rows of those
        // keys: A steps 32 bytes inside P's swizzled rows; B is the CTA's
        // value column blocks of that range (adjacent ring slots, 8 KB apart:
        // the N extent) and steps two 8-key groups (2 KB) down them.  The
        // group's slots are released once its products complete.
#pragma unroll
        for (int q = 0; q < kDv / 256; ++q) {
          const int sl = s0 + C::kVGroup * q < kRingV ? s0 + C::kVGroup * q
                                                      : s0 + C::kVGroup * q - kRingV;
          const uint64_t bd =
              smem_desc(sb + C::kOffV + uint32_t(sl) * kVSlotBytes, kVSlotBytes, 1024, kSwizzle128B);
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k)
            mma_ss_any<kPair>(tmem + uint32_t(256 * q), ad0 + uint64_t((uint32_t(k) * 32u) >> 4),
                              bd + uint64_t((uint32_t(k) * 2048u) >> 4), idesc,
                              (t > 0 || k > 0) ? 1u : 0u);
#pragma unroll
          for (int g = 0; g < C::kVGroup; ++g) commit_local<kPair>(bar(C::B_EMPTY + sl + g), C::kPvMask);
        }
        // re-arm the buffer for tile t + kPBufs before its release reaches
        // the QK CTA (the release follows this product's completion)
        if (lane == 0 && t + kPBufs < ntiles) mbar_arrive_expect_tx(bar(C::B_PFULL + bs), kPPayload);
        __syncwarp();
        commit_mc<kPair>(bar(C::B_PFREE + bs), C::kQkMask);
        if (lane == 0) VA_TRACE_EVENT(4, 1, t);
        VA_PH(2);
      }
      if (lane == 0) VA_PH_STORE(10);
      // last command to the row warps: no more rescales
      if (lane == 0) {
        *cmd = kCmdDone;
        mbar_arrive(bar(C::B_OGO));
        if constexpr (kPair) {
          st_cluster_u32(m_cmd, kCmdDone);
          mbar_arrive_remote(m_ogo);
        }
      }
      __syncwarp();
      commit_local<kPair>(bar(C::B_MMAFIN), C::kPvMask);
      mbar_wait(bar(C::B_MMAFIN), 0, nullptr, kWaitCycles);
      __syncwarp();
      if constexpr (!kPair) cluster_arrive_relaxed();   // the releases to the QK CTA precede MMAFIN
    } else if (warp == 1) {
      // ---- odd rank of the PV pair: forwards each tile's arrivals -- its
      // value blocks and its P buffer -- to the even rank in one arrival (a
      // cluster-scope release costs about 1100 cycles, so one per tile), and
      // re-arms its own P buffers
      const uint32_t fullp = mapa(bar(C::B_FULLP), mate);
      const uint32_t peer_any = mapa(sb + C::kOffPeerAny, mate);
      if (lane == 0)
        for (int t = 0; t < kPBufs && t < ntiles; ++t)
          mbar_arrive_expect_tx(bar(C::B_PFULL + t), kPPayload);
      __syncwarp();
      for (int t = 0; t < ntiles; ++t) {
        const int fi = t % C::kFullRing;
        const int bs = t % kPBufs;
        const bool got =
            mbar_wait(bar(C::B_FULL + fi), uint32_t(t / C::kFullRing) & 1u, abort_flag,
                      kWaitCycles) &&
            mbar_wait<true>(bar(C::B_PFULL + bs), uint32_t(t / kPBufs) & 1u, abort_flag,
                            kWaitCycles);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) fail();
          break;
        }
        fence_proxy_async_cta();   // this CTA's cp.async writes, read by the pair's tensor core
        // whether any of this CTA's rows rescales at this tile, for the even
        // rank's issuer (published by the release arrival below); the buffer
        // is re-armed before the even rank's products -- and so the release
        // of this buffer to the QK CTA -- can follow
        if (lane == 0) {
          const volatile uint32_t* fl = reinterpret_cast<const volatile uint32_t*>(
              gb + C::kOffP + uint32_t(bs) * kPBufBytes + kPFlags);
          st_cluster_u32(peer_any + 4u * uint32_t(bs), (fl[0] | fl[1] | fl[2] | fl[3]) & 1u);
          if (t + kPBufs < ntiles) mbar_arrive_expect_tx(bar(C::B_PFULL + bs), kPPayload);
          mbar_arrive_remote(fullp + 8u * uint32_t(fi));
        }
        __syncwarp();
      }
      // the even rank's products read this CTA's shared memory and write its
      // tensor memory until their last commit
      (void)mbar_wait(bar(C::B_MMAFIN), 0, nullptr, kWaitCycles);
      __syncwarp();
    } else if (warp >= 4) {
      // ---- row warps: rescale O rows on command, then the split's partial;
      // warpgroup `half` owns columns [256*half, 256*half + 256)
      const int r = q4 * 32 + lane;
      const int lr = row0 + r;
      const bool row_ok = lr < R;
      const uint32_t tl = tmem + (uint32_t(q4 * 32) << 16) + 256u * uint32_t(half);
      const uint32_t ocorr_issuer = kPair ? mapa(bar(C::B_OCORR), mate) : 0u;
      bool ok = true;
      for (uint32_t k = 0;; ++k) {
        const bool go = mbar_wait<kPair>(bar(C::B_OGO), k & 1u, abort_flag, kWaitCycles);
        if (!__all_sync(0xffffffffu, go)) {
          fail();
          ok = false;
          break;
        }
        const uint32_t c = *cmd;
        if (c == kCmdDone) break;
        const float a = reinterpret_cast<const float*>(gb + C::kOffP + c * kPBufBytes + kPAlpha)[r];
        tc_fence_after();
        // tcgen05.ld/st are warp-collective: the whole warp takes part when
        // any of its rows rescales, each lane scaling by its own factor
        if (__any_sync(0xffffffffu, a != 1.f)) {
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t v[32];
            tmem_ld32(tl + 32u * uint32_t(cc), v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * a);
            tmem_st32(tl + 32u * uint32_t(cc), v);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        if (!kPair || issuer_cta) {
          mbar_arrive(bar(C::B_OCORR));
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(ocorr_issuer);
        }
      }
      const bool fin = ok && mbar_wait<true>(bar(C::B_FIN), 0, abort_flag, kWaitCycles) &&
                       mbar_wait(bar(C::B_MMAFIN), 0, abort_flag, kWaitCycles);
      // all row warps agree before the staged write-out below
      const bool go = named_sync_and(kSoftmaxBar, kSoftmax, __all_sync(0xffffffffu, fin));
      if constexpr (!kPair) cluster_arrive_relaxed();   // FIN received: the QK CTA writes here no more
      if (go) {
        if (tid == 128) VA_TRACE_CTA(7, 5);
        tc_fence_after();
        // The split's partial (128 rows x 512, normalised by the row sum,
        // rounded to bf16) leaves through shared memory and the bulk-copy
        // engine, one 512-byte half row per copy: the P and value buffers are
        // idle now and hold all 128 padded rows.
        const float inv = reinterpret_cast<const float*>(gb + C::kOffFin)[r];
        uint8_t* stg = gb + C::kOffP;
        uint8_t* rowp = stg + r * kEpiRowBytes + 512 * half;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32];
          tmem_ld32(tl + 32u * uint32_t(c), v);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(v[2 * e]) * inv,
                                                           __uint_as_float(v[2 * e + 1]) * inv);
            pk[e] = *reinterpret_cast<const uint32_t*>(&h);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(rowp + 64 * c + 16 * j) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
        fence_proxy_async_cta();   // staged half row, read by this thread's bulk copy
        if (tid == 128) VA_TRACE_CTA(5, 0);
        // each thread sends its own half row as soon as it is staged, and
        // waits only until the copy has read it (the writes complete before
        // the grid does)
        if (row_ok)
          bulk_store_global(p.part_o + (size_t(split) * rows_total + size_t(b) * R + lr) * kDv + 256 * half,
                            smem_u32(rowp), 512u);
        bulk_commit();
        bulk_wait_read<0>();
        if (lane == 0 && warp == 4) VA_TRACE_CTA(5, 1);
      } else if (ok && !fin) {
        fail();
      }
    }
  }

  if (tid == 0) VA_TRACE_CTA(trace_role, 2);
  tc_fence_before();
  __syncthreads();
  if (tid == 0) *flag_word = *cta_flags;   // this CTA's status bits
  if (tid == 0) VA_TRACE_CTA(trace_role, 3);
  if constexpr (kPair) {
    // Every CTA of the cluster has finished every role before any frees its
    // tensor memory or leaves: a pair's products read and write both CTAs'
    // memories, and the odd ranks' forwarded arrivals land in the even ranks.
    cluster_sync();
    if (warp == 2) {
      tc_fence_after();
      tmem_dealloc_pair(tmem, kTmemCols);
    }
  } else {
    if (warp == 2) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
    // Neither CTA leaves while the other may still touch its shared memory.
    // The PV CTA's threads arrived once they were done with the QK CTA: its
    // producers after their last copy, its MMA warp after the last products
    // (whose P-buffer releases reach the QK CTA, which waits for them itself),
    // its row warps once the QK CTA's row sums had landed.  So the QK CTA
    // leaves during the PV CTA's write-out, and the PV CTA, arrived already,
    // only waits here for the QK CTA to have arrived.
    if (rank == 0)
      cluster_sync();
    else
      cluster_wait();
  }
  if (tid == 0) VA_TRACE_CTA(trace_role, 4);
}

// Clusters of `ctas` CTAs of the kernel that the device runs at once.
template <bool kPair>
int max_clusters() {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(unsigned(Cfg<kPair>::kCtas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg<kPair>::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(Cfg<kPair>::kCtas);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, partial_tc_kernel<kPair>, &cfg) != cudaSuccess) {
    n = 0;
    (void)cudaGetLastError();
  }
  return n;
}

}  // namespace

bool tc_supported(int, int, int) { return true; }

// Two-SM products pay off once a request has more than one 128-row block; a
// caller can ask for the one-SM shape at any row count (VA_PATH_TC_1SM).
bool tc_use_pair(int T, int H, int flags) {
  return flags != VA_PATH_TC_1SM && long(T) * H > kRows;
}

// Splits per (row unit, request).  `clusters` is the number of clusters of
// the chosen shape the device runs at once (clusters live inside one GPC, so
// GPCs whose SM count is not a multiple of the cluster size strand SMs).
// With few (row unit, request) items, one wave of clusters splits each item
// evenly.  With many (more than half a wave), one split per item would leave
// clusters idle and let the longest request of a ragged batch set the time,
// so the items are split into a few waves of clusters instead: about five and
// a half for the one-SM shape, five for the pair shape (measured on 8
// requests at H=64 with prefixes from 13k to 46k keys: one-SM shape, 3, 4,
// 5, 6, 7, 8, 10 splits per item -> 727, 734, 693, 691, 669, 678, 700 us per
// step; pair shape, 4 .. 10 -> 561, 555, 546, 561, 568, 565, 589 us).
// (Prefix lengths live on the device, so the rule uses the shape only; splits
// past a request's keys exit at once.)
int tc_auto_nsplit(int B, int T, int H, int clusters, bool pair) {
  const long unit = pair ? 2 * kRows : kRows;
  const long units = (long(T) * H + unit - 1) / unit;
  const long items = units * B;
  const long waves2 = pair ? 10 : 11;   // twice the target number of waves
  long ns = 2 * items <= clusters ? clusters / items
                                  : (waves2 * clusters + 2 * items - 1) / (2 * items);
  if (ns < 1) ns = 1;
  if (ns > VA_NSPLIT_MAX) ns = VA_NSPLIT_MAX;
  return int(ns);
}

// 128-row blocks of status words per request: the grid's units x their blocks.
int tc_flag_blocks(int T, int H, bool pair) {
  const int unit = pair ? 2 * kRows : kRows;
  return ceil_div(T * H, unit) * (unit / kRows);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t init_partial_tc(int* max_pairs, int* max_quads) {
  cudaError_t e = cudaFuncSetAttribute(partial_tc_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(Cfg<false>::kSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(partial_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(Cfg<true>::kSmemBytes));
  if (e != cudaSuccess) return e;
  *max_pairs = max_clusters<false>();
  *max_quads = max_clusters<true>();
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess && fn)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return cudaSuccess;
}

// Tensor maps of a contiguous pool: 3-D (64 columns, pool rows, column
// blocks: strides one row and 128 bytes), a box of `rows` keys x `blocks`
// column blocks covering a CTA's share of a 64-key tile; 2-D (576 columns,
// pool rows; blocks = 0), a box of one column block of `rows` keys.
bool encode_pool_map(CUtensorMap* m, const Params& p, int blocks, int rows) {
  if (blocks > 0) {
    cuuint64_t dims[3] = {64u, cuuint64_t(p.num_slots), cuuint64_t(kKBlocks)};
    cuuint64_t strides[2] = {cuuint64_t(p.kv_stride) * 2u, 128u};
    cuuint32_t box[3] = {64u, uint32_t(rows), uint32_t(blocks)};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(p.kv), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  cuuint64_t dims[2] = {cuuint64_t(kDqk), cuuint64_t(p.num_slots)};
  cuuint64_t strides[1] = {cuuint64_t(p.kv_stride) * 2u};
  cuuint32_t box[2] = {64u, uint32_t(rows)};
  cuuint32_t estr[2] = {1u, 1u};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(p.kv), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of the queries: 3-D (64 features, query rows B*T*H, column
// blocks: strides one 1152-byte row and 128 bytes); a box of 64 rows x 9
// blocks is half a row block's Q.
bool encode_q_map(CUtensorMap* m, const Params& p) {
  cuuint64_t dims[3] = {64u, cuuint64_t(p.B) * cuuint64_t(p.rows_per_req), cuuint64_t(kKBlocks)};
  cuuint64_t strides[2] = {cuuint64_t(kDqk) * 2u, 128u};
  cuuint32_t box[3] = {64u, 64u, uint32_t(kKBlocks)};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(p.q), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_partial_tc(const Params& p, int /*num_sms*/, cudaStream_t st) {
  const bool pair = p.tc_pair != 0;
  const int ctas = pair ? Cfg<true>::kCtas : Cfg<false>::kCtas;
  const int unit = pair ? Cfg<true>::kUnitRows : Cfg<false>::kUnitRows;
  // Contiguous pools are read with TMA box loads; the maps are encoded on the
  // host for this call's pool.  Paged calls do not use them.  Pair shares: a
  // QK CTA's 32 keys of a tile (3-D box of 9 blocks, 2-D box per block where
  // the ring wraps); a PV CTA's value blocks, two boxes of 2 blocks x 64 keys.
  CUtensorMap tk, tv, t2, tq;
  memset(&tk, 0, sizeof tk);
  memset(&tv, 0, sizeof tv);
  memset(&t2, 0, sizeof t2);
  if (!g_encode || !encode_q_map(&tq, p)) return cudaErrorNotSupported;
  int box3d = 0;
  if (p.kv_start) {
    const int krows = pair ? Cfg<true>::kSlotKeys : kTile;
    if (!encode_pool_map(&t2, p, 0, krows)) return cudaErrorNotSupported;
    if (encode_pool_map(&tk, p, kKBlocks, krows) &&
        encode_pool_map(&tv, p, pair ? 2 : kVBlocks, kTile))
      box3d = 1;
  }
  // A programmatic dependent of the stream's previous kernel (programmatic
  // stream serialization): after the draft-row append kernel the clusters
  // run while it does (see the producers' griddepcontrol.wait); as the call's
  // first kernel they may start while the stream's previous kernel finishes
  // and wait for it before reading any input.
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(unsigned(ctas * p.nsplit), unsigned(ceil_div(p.rows_per_req, unit)),
                     unsigned(p.B));
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = pair ? Cfg<true>::kSmemBytes : Cfg<false>::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(ctas);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return pair ? cudaLaunchKernelEx(&cfg, partial_tc_kernel<true>, p, tk, tv, t2, tq, box3d)
              : cudaLaunchKernelEx(&cfg, partial_tc_kernel<false>, p, tk, tv, t2, tq, box3d);
}

}  // namespace va
