// gemm_kernel.cuh -- persistent, warp-specialized tcgen05 GEMM for sm_103a.
//
//   C[M,N] = A[M,K] x B[N,K]^T, fp16 in, fp32 or fp16 accumulate, fp16 out
//   (tilus "A Minimal Hopper Matmul", section "Block Tiling").
//
// One template, five forms:
//   kCtas = 1           one CTA per SM owns a 128 x kBN tile of C (kBN = 64..256);
//   kCtas = 2           a cluster of two CTAs on neighbouring SMs owns a
//                       256 x kBN tile: each CTA loads its 128 rows of A and
//                       half of the tile's rows of B, and one thread of the
//                       leader CTA issues tcgen05.mma.cta_group::2 (M = 256)
//                       over both CTAs' shared memory, so every SM stages a
//                       third less operand data per FLOP (at kBN = 256);
//   kCtas = 2, kMc = 2  a cluster of four CTAs: two such pairs on neighbouring
//                       tiles of one tile-row, each CTA loading half of its
//                       pair's A rows and multicasting them into both pairs
//                       (for rows whose pitch is not a multiple of 128 bytes,
//                       where every TMA row straddles two L2 lines);
//   kSwap               roles swapped for C with few rows: the MMA's M runs
//                       over 128 columns of C (rows of B) and its N over
//                       kBN = 16..64 rows of C, and the epilogue transposes
//                       8 x 8 blocks in registers and writes C straight from
//                       them, 16 bytes per lane;
//   kSplit = 2 or 4     a cluster of single CTAs (plain or swapped roles)
//                       shares every tile it is given, each CTA accumulating
//                       one k-slice, and the partial tiles meet in shared
//                       memory -- for problems of few tiles with many
//                       k-blocks each, without a round trip through global
//                       memory.  Plain roles: the CTAs of rank > 0 write
//                       their fp32 partials into rank 0's shared memory
//                       (st.shared::cluster, one release arrival per thread)
//                       and rank 0 adds them to its own, in rank order, and
//                       stores the tile.  Swapped roles (kSplit = 2): each
//                       CTA finishes half of the tile's rows of C and sends
//                       the other half of its partial to the other CTA
//                       (st.async, bytes completed on the receiver's
//                       barrier).
// Operands are K-contiguous or M/N-contiguous (run-time choice: TMA box shape,
// shared-memory descriptor and the instruction descriptor's transpose bits).
//
// Units (CTAs, pairs or four-CTA clusters) are persistent.  Their work list
// (Sched) is a share of the part-empty last wave's tiles cut into equal
// k-block ranges (stream-K) followed by whole tiles over a grouped raster,
// dealt round robin or, for long runs of waves, in a dynamic order taken
// from a global ticket counter.  A tile shared by several units is finished
// by whichever contributes last: the others park fp32 partials in a
// workspace, and the last one sums them in unit order.  Inside a CTA the work
// is split by warp, after the producer / consumer split of tilus "Warp
// Specialization", redesigned for tcgen05:
//
//   warps 0 and 6    TMA producers: a kStages-deep ring of k-blocks, warp 0
//                    loading A and warp 6 loading B.
//   warp 1           allocates tensor memory (TMEM); in the leader CTA it
//                    issues every tcgen05.mma and releases each stage with
//                    tcgen05.commit onto its "empty" mbarrier(s).
// Producers and issuer run as whole, converged warps with one elected lane
// issuing: measured on GB300, a lone divergent lane spends ~486 cycles per
// k-block on 4 MMAs, a commit and a barrier test, a converged warp ~322; with
// a 256-wide tile the tensor pipe needs 512 cycles per k-block, so only the
// converged form keeps it fed.
//   warps 2..5       epilogue: tcgen05.ld the accumulator, round to fp16,
//                    stage through swizzled shared memory, TMA-store.
//   warp 7           tile scheduler of the dynamic order (cluster leader only;
//                    idle otherwise).
//
// The accumulator is double-buffered in TMEM (2 x kBN columns), so the
// epilogue of one work item overlaps the main loop of the next; tmem_full /
// tmem_empty barriers hand the buffers back and forth.
//
// Every wait is bounded: a wait that outlives the timeout records the site in
// a device watchdog word and raises the CTA's abort flag; every role then
// leaves its loop, the CTA waits (again bounded) for its own loads and MMAs,
// frees tensor memory and returns.
#pragma once
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace gb300 {

// Where a wait gave up (reported in the watchdog record's second word).
enum WaitSite : uint32_t {
  kSiteEmpty = 1,      // producer waiting for a free stage
  kSiteFull = 2,       // MMA issuer waiting for a filled stage
  kSiteTmemEmpty = 3,  // MMA issuer waiting for a drained accumulator buffer
  kSiteTmemFull = 4,   // epilogue waiting for a finished accumulator
  kSiteMmaDone = 5,    // teardown: waiting for the last MMAs
  kSiteDrain = 6,      // teardown: producer waiting for its last stages
  kSiteTileFull = 7,   // a role waiting for the next tile from the tile scheduler
  kSiteTileEmpty = 8,  // the tile scheduler waiting for a free slot of its ring
  kSiteRedFull = 9,    // split-K leader waiting for the other CTAs' partial tiles
  kSiteRedEmpty = 10,  // split-K CTA waiting for the leader to free its partial slot
};

constexpr uint32_t kStatusTimeout = 5;  // == GEMM_ERR_TIMEOUT

struct GemmArgs {
  int32_t M, N, K;
  int32_t tiles_m, tiles_n, num_kb, num_tiles;
  int32_t group_m;      // raster group height, in tiles
  uint32_t* err;        // device watchdog record, 4 words
  uint64_t timeout_ns;  // longest allowed single wait
  int32_t skip_kb;      // fault injection, -1 = off
  // Operand layouts: 0 = K contiguous (A [M,K], B [N,K]); 1 = M (resp. N)
  // contiguous (A stored [K,M], B stored [K,N]); loaded as 64 x 64 boxes.
  int32_t a_mn, b_mn;
  // Schedule: tiles [0, dp_tiles) are dealt out whole, round robin over the
  // units (CTAs or CTA pairs).  The remaining tiles form the stream-K tail:
  // their sk_iters = (num_tiles - dp_tiles) * num_kb k-blocks are cut into
  // sk_units equal contiguous ranges, so a tail tile may be shared by several
  // units, each accumulating a k-range of it.
  int32_t dp_tiles;
  int32_t sk_units;     // 0 = no stream-K tail
  int64_t sk_iters;
  float* sk_ws;         // partial accumulators: [unit][2 slots][CTA of unit][128 x 256] fp32
  uint32_t* sk_count;   // per tail tile and CTA of the tile: contributions so far (self-resetting)
  uint16_t* C;          // output (fp16 bits), row pitch ldc elements: the swapped-roles
  int64_t ldc;          // epilogue stores directly
  // Dynamic order of whole tiles: [0] tickets taken, [1] units finished (both
  // back to zero when a launch ends).  nullptr: the static round robin.
  uint32_t* tile_ctr;
  // Clock record, or nullptr: CTA 0 adds 1, its lifetime in SM cycles
  // (%clock64) and in ns (%globaltimer) to [0], [1], [2], so the host can
  // read the SM clock the kernel actually ran at.
  unsigned long long* clk;
};

struct Watch {
  volatile uint32_t* abort;
  uint32_t* err;
  uint64_t timeout_ns;
};

// Slow path of a bounded mbarrier wait.  Returns false when the wait gave up,
// either because the CTA is aborting (and honor_abort) or after timeout_ns.
template <bool kClusterScope>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, Watch w, uint32_t site,
                                       int32_t tile, bool honor_abort) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    const bool done = kClusterScope ? ptx::mbar_try_wait_cluster(bar, parity)
                                    : ptx::mbar_try_wait(bar, parity);
    if (done) return true;
    if (honor_abort && *w.abort) return false;
    if (ptx::globaltimer_ns() - t0 > w.timeout_ns) {
      if (atomicCAS(w.err, 0u, kStatusTimeout) == 0u) {
        w.err[1] = site;
        w.err[2] = blockIdx.x;
        w.err[3] = static_cast<uint32_t>(tile);
      }
      *w.abort = 1u;
      return false;
    }
  }
}

template <bool kClusterScope>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Watch& w,
                                         uint32_t site, int32_t tile, bool honor_abort = true) {
  const bool done =
      kClusterScope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
  if (done) return true;
  return wait_slow<kClusterScope>(bar, parity, w, site, tile, honor_abort);
}

// Warp-collective wait: every lane waits and the warp agrees on the outcome,
// so the code after it stays converged.  The producer and MMA roles run as
// whole warps and let one elected lane issue: values computed in converged
// code stay warp-uniform, and both the issue of tcgen05.mma / TMA and the
// barrier test cost far fewer cycles than from a lone divergent lane.
template <bool kClusterScope>
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const Watch& w,
                                              uint32_t site, int32_t tile,
                                              bool honor_abort = true) {
  return __all_sync(0xffffffffu, wait_bar<kClusterScope>(bar, parity, w, site, tile, honor_abort));
}

// One piece of work for a unit: k-blocks [kb0, kb1) of one output tile.
struct WorkItem {
  int32_t tile;        // linear tile index, before rastering
  int32_t kb0, kb1;
  int32_t sk_tile;     // index in the stream-K tail, -1 for a whole tile
  int32_t splits;      // units contributing to this tile (1: no fix-up)
  int32_t first_unit;  // first contributing unit (stream-K tail only)
};

// Where a role reads the dynamic tile order: a two-slot ring in its own
// CTA's shared memory, filled by the unit's tile scheduler (tile_full[i]
// completes when slot i holds the next tile), and emptied by arriving on
// tile_empty[i] in the leader CTA of the cluster.  Every consumer warp reads
// every slot, in order.
struct TileRing {
  uint32_t slot0;   // this CTA: slot i at slot0 + 4 i
  uint32_t full0;   // this CTA: tile_full[i] at full0 + 8 i
  uint32_t empty0;  // the cluster's leader CTA: tile_empty[i] at empty0 + 8 i
  Watch w;
  bool cluster;     // the kernel runs in clusters (addresses are cluster-wide)
  uint32_t took;    // nonzero for the leader's A producer: it arrives here on each read,
                    // which tells the scheduler to take the next ticket
};

// The work list of one unit, identical in every role of the unit's CTAs:
// first its share of the stream-K tail, then its whole tiles.  Whole tiles
// come round robin (tile unit, unit + units, ...) in the static order; in
// the dynamic order (tile_ctr set) the first is still tile `unit` and the
// rest are the tiles the unit's scheduler takes from a global ticket
// counter as the unit needs them, so tiles start in order across units and
// the tiles in flight stay within about one wave however far units drift
// apart (operands then stay in L2 between their uses by neighbouring tiles).
struct Sched {
  int32_t unit, units, dp_tiles, num_kb, sk_units;
  int32_t kslice, kslices;  // split-K clusters: this CTA's k-slice of every tile, of kslices
  int64_t sk_iters;
  int32_t next_dp;
  int64_t x, x_end;  // this unit's remaining range of tail k-blocks
  bool dyn;          // dynamic order of whole tiles after the first
  bool first_done;   // the unit's first whole tile has been handed out
  int32_t n;         // ring slots read so far
  TileRing ring;

  __device__ __forceinline__ Sched(const GemmArgs& a, int32_t unit_, int32_t units_,
                                   const TileRing& ring_ = TileRing{}, int32_t kslice_ = 0,
                                   int32_t kslices_ = 1)
      : unit(unit_), units(units_), dp_tiles(a.dp_tiles), num_kb(a.num_kb),
        sk_units(a.sk_units), kslice(kslice_), kslices(kslices_), sk_iters(a.sk_iters),
        next_dp(unit_), x(0), x_end(0),
        dyn(a.tile_ctr != nullptr), first_done(false), n(0), ring(ring_) {
    if (sk_units > 0 && unit < sk_units) {
      x = bound(unit);
      x_end = bound(unit + 1);
    }
  }
  // The next tile from the scheduler's ring, or -1 when there are no more
  // (or the wait gave up).  Called by whole, converged warps; lane 0 frees
  // the slot, once the slot's value has been read.
  __device__ __forceinline__ int32_t ring_read() {
    const int i = n & 1;
    const uint32_t par = static_cast<uint32_t>((n >> 1) & 1);
    ++n;
    const bool ok =
        ring.cluster ? wait_bar_warp<true>(ring.full0 + 8u * i, par, ring.w, kSiteTileFull, -1)
                     : wait_bar_warp<false>(ring.full0 + 8u * i, par, ring.w, kSiteTileFull, -1);
    const uint32_t v = ok ? ptx::ld_shared_u32(ring.slot0 + 4u * i) : 0xffffffffu;
    if ((threadIdx.x & 31) == 0) {
      if (ring.cluster)
        ptx::mbar_arrive_relaxed_cluster_after(ring.empty0 + 8u * i, v);
      else
        ptx::mbar_arrive_relaxed_cta_after(ring.empty0 + 8u * i, v);
      if (ring.took) ptx::mbar_arrive_relaxed_cta_after(ring.took, v);
    }
    return static_cast<int32_t>(v);
  }
  // A whole tile; in a split-K cluster, this CTA's k-slice of it (the
  // slices of a tile's kslices CTAs partition its k-blocks, each non-empty).
  __device__ __forceinline__ void whole(WorkItem& w, int32_t t) const {
    w.tile = t;
    w.kb0 = kslice * num_kb / kslices;
    w.kb1 = (kslice + 1) * num_kb / kslices;
    w.sk_tile = -1;
    w.splits = kslices;
    w.first_unit = unit;
  }
  // First tail k-block of unit u.
  __device__ __forceinline__ int64_t bound(int64_t u) const { return u * sk_iters / sk_units; }
  // The unit whose range holds tail k-block `it` (the largest u with bound(u) <= it).
  __device__ __forceinline__ int32_t unit_of(int64_t it) const {
    return static_cast<int32_t>(((it + 1) * sk_units - 1) / sk_iters);
  }
  // Workspace slot unit u uses for tail tile t: 0 if t is the first tile its
  // range touches, else 1 (only a range's first and last tiles can be partial).
  __device__ __forceinline__ int32_t slot_of(int32_t u, int32_t t) const {
    return static_cast<int32_t>(bound(u) / num_kb) == t ? 0 : 1;
  }
  // Whether next() may hand out another item (with the dynamic order, whose
  // next tile is not known yet, always true once the first whole tile is out).
  __device__ __forceinline__ bool has_more() const {
    if (x < x_end) return true;
    if (dyn && first_done) return true;
    return next_dp < dp_tiles;
  }
  // Stream-K pieces come first and whole tiles after them: the fix-up of a
  // shared tile (reading the other units' partials) then overlaps the main
  // loop of a later whole tile instead of ending the kernel.
  __device__ __forceinline__ bool next(WorkItem& w) {
    if (x >= x_end) {
      if (dyn && first_done) {
        const int32_t t = ring_read();
        if (t < 0) return false;
        whole(w, t);
        return true;
      }
      first_done = true;
      if (next_dp >= dp_tiles) return false;
      whole(w, next_dp);
      next_dp += units;
      return true;
    }
    if (x < x_end) {
      const int32_t t = static_cast<int32_t>(x / num_kb);
      const int64_t t0 = static_cast<int64_t>(t) * num_kb, t1 = t0 + num_kb;
      const int64_t e = x_end < t1 ? x_end : t1;
      w.tile = dp_tiles + t;
      w.kb0 = static_cast<int32_t>(x - t0);
      w.kb1 = static_cast<int32_t>(e - t0);
      w.sk_tile = t;
      w.first_unit = unit_of(t0);
      w.splits = unit_of(t1 - 1) - w.first_unit + 1;
      x = e;
      return true;
    }
    return false;
  }
};

// Tile configuration.  kCtas CTAs cooperate on one tile of kTileM x kBN.
template <int kCtas_, int kStages_, bool kAccF16_, int kBN_ = 256, bool kSwap_ = false,
          int kMc_ = 1, int kSplit_ = 1>
struct GemmCfg {
  static constexpr int kCtas = kCtas_;
  // kMc = 2: a cluster holds two CTA pairs working on neighbouring tiles of
  // the same tile-row; the pairs share the tile-row's A block, each CTA
  // loading half of its 128 rows and multicasting it to the CTA in the same
  // position of the other pair, so every SM requests half as many A bytes.
  static constexpr int kMc = kMc_;
  static constexpr int kPairs = kMc;  // CTA pairs (or lone CTAs) per cluster
  // kSplit > 1: a cluster of kSplit single CTAs shares every tile it is
  // given, each CTA accumulating its own k-slice.  Plain roles: the CTAs of
  // rank > 0 write their fp32 partial tiles into the shared memory of rank 0,
  // which adds them to its own (in rank order) and stores the tile.  Swapped
  // roles (kSplit = 2): rank r finishes accumulator columns [r kBN/2,
  // (r+1) kBN/2) (rows of C) and receives the other rank's partial of them.
  static constexpr int kSplit = kSplit_;
  static constexpr int kClusterCtas = kCtas * kPairs * kSplit;
  // Swapped roles (for small M): the MMA's "A" operand is a 128-row tile of B
  // and its "B" operand a kBN-row tile of A, so D = tile of C^T.
  static constexpr bool kSwap = kSwap_;
  static constexpr int kBM = 128;                 // rows of C per CTA
  static constexpr int kBN = kBN_;                // columns of C per tile
  static constexpr int kBK = 64;                  // K per stage (one 128-byte swizzle row)
  static constexpr int kTileM = kBM * kCtas;      // rows of C per tile (of one pair)
  static constexpr int kBRows = kBN / kCtas;      // rows of B each CTA loads
  static constexpr int kStages = kStages_;
  static constexpr bool kAccF16 = kAccF16_;
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = kBRows * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;  // landed in each CTA per stage
  static constexpr int kTxBytes = kStageBytes * kCtas;   // counted on the leader's barrier
  static constexpr int kEpiWarps = 4;
  static constexpr int kEpiBufBytes = 32 * 128;  // 32 rows x 64 fp16, 128B swizzle
  static constexpr int kEpiBytes = kSwap ? 0 : kEpiWarps * 2 * kEpiBufBytes;
  // Split-K: the fp32 partials a CTA receives, each stored
  // [column / 4][row][column % 4]: kSplit - 1 whole 128 x kBN tiles (rank 0,
  // plain roles) or one 128 x kBN/2 half (every rank, swapped roles).
  static constexpr int kRedBytes = kSwap ? (kSplit - 1) * kBM * (kBN / kSplit) * 4
                                         : (kSplit - 1) * kBM * kBN * 4;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kStages * kABytes;
  static constexpr int kOffEpi = kStages * kStageBytes;
  static constexpr int kOffRed = kOffEpi + kEpiBytes;
  static constexpr int kOffBar = kOffRed + kRedBytes;
  // full, empty, tmem_full[2], tmem_empty[2], mma_done, tile_full[2], tile_empty[2],
  // tile_took, red_full, red_empty
  static constexpr int kNumBars = 2 * kStages + 12;
  static constexpr int kOffSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffSlot + 4;
  static constexpr int kOffFlag = kOffAbort + 4;           // stream-K "last contributor" flag
  static constexpr int kOffTiles = kOffFlag + 4;           // tile ring: two slots
  static constexpr int kSmemBytes = kOffTiles + 8 + 1024;  // + slack to align the base to 1024
  static constexpr int kPartialFloats = kBM * kBN;         // one CTA's share of a partial tile
  static constexpr int kTmemCols = 2 * kBN;
  static constexpr int kWarpProducerB = 6;  // warps 0 and 6 load A and B
  static constexpr int kWarpSched = 7;      // tile scheduler (dynamic order, leader CTA)
  static constexpr int kThreads = 256;
  // Warps that read the tile ring: in every CTA both producers and the four
  // epilogue warps, and the MMA issuer in each pair's (or lone CTA's) leader.
  static constexpr int kTileConsumers = kClusterCtas * (2 + kEpiWarps) + (kCtas == 1 ? 1 : kPairs);
  static constexpr uint32_t kIdesc = ptx::idesc_f16(kTileM, kBN, !kAccF16);

  static_assert(kCtas == 1 || kCtas == 2, "one CTA or a CTA pair");
  static_assert(kMc == 1 || (kMc == 2 && kCtas == 2 && !kSwap),
                "A multicast between two CTA pairs only");
  static_assert(kClusterCtas <= 8, "portable cluster size");
  static_assert(kSplit == 1 || ((kSplit == 2 || kSplit == 4) && kCtas == 1 && kMc == 1 && !kAccF16),
                "split-K clusters: 2 or 4 single CTAs, fp32 partials");
  static_assert(!kSwap || kSplit <= 2, "swapped roles split K in two (a half tile per CTA)");
  static_assert(kSwap ? (kCtas == 1 && (kBN == 16 || kBN == 32 || kBN == 64))
                      : (kBN == 64 || kBN == 128 || kBN == 256),
                "tile width: 64, 128 or 256; 16, 32 or 64 with swapped roles (one CTA)");
  static_assert(kBRows >= 8 && kBRows % 8 == 0, "B rows per CTA: whole 8-row swizzle atoms");
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
                "TMEM is allocated in powers of two from 32 to 512 columns");
  static_assert(kSmemBytes <= 232448, "exceeds 227 KB of shared memory per CTA");
  static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "swizzle atoms need 1024 B alignment");
  // Barriers sit after every TMA destination, never inside one (tilus "A
  // Minimal Hopper Matmul", Epilogue note: a barrier placed inside a live TMA
  // destination is silently corrupted).
  static_assert(kOffBar >= kOffRed + kRedBytes, "barriers overlap a TMA or partial buffer");
};

// Grouped raster: tiles are walked down a group of `group` tile-rows before
// moving one tile-column right, so tiles in flight at the same time share A
// rows and B rows in L2.  A bijection of [0, tiles_m*tiles_n).
__device__ __forceinline__ void raster(int32_t t, int32_t tiles_m, int32_t tiles_n, int32_t group,
                                       int32_t& mb, int32_t& nb) {
  const int32_t per = group * tiles_n;
  const int32_t g = t / per;
  const int32_t m0 = g * group;
  const int32_t gs = min(group, tiles_m - m0);
  const int32_t r = t - g * per;
  mb = m0 + r % gs;
  nb = r / gs;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// kCols consecutive fp32 accumulator columns of this thread's TMEM lane
// (32x32b loads: thread t of the warp reads lane base + t), one wait for all.
template <int kCols>
__device__ __forceinline__ void tmem_ld_f32(uint32_t taddr, float* out) {
  static_assert(kCols % 8 == 0, "columns come in groups of eight");
  uint32_t v[kCols];
#pragma unroll
  for (int g = 0; g < kCols / 16; ++g)
    ptx::tmem_ld_32x32b_x16(taddr + g * 16, *reinterpret_cast<uint32_t(*)[16]>(v + g * 16));
  if constexpr (kCols % 16 != 0)
    ptx::tmem_ld_32x32b_x8(taddr + kCols / 16 * 16,
                           *reinterpret_cast<uint32_t(*)[8]>(v + kCols / 16 * 16));
  ptx::tmem_wait_ld(v);
#pragma unroll
  for (int i = 0; i < kCols; ++i) out[i] = __uint_as_float(v[i]);
}

// Store kRows rows of a swapped-roles tile of C.  Lane l of the warp holds
// column n_lane of C (the lanes' columns consecutive, the first a multiple
// of 8) and in v[i] the value of row m0 + i.  Within each group of eight
// lanes, every 8 x 8 block (eight rows, the group's eight columns) is
// transposed in registers by a three-step butterfly: at distance d = 4, 2, 1
// a lane swaps with lane ^ d the four values whose index differs from its
// own lane index in bit d.  Each step runs over all blocks before the next,
// so its shuffles are independent and issue back to back.  After it lane
// (g, j) holds row 8b + j, columns 8g .. 8g + 7 of the warp's 32, rounded to
// fp16 and written as one 16-byte store: per row the warp's four groups
// write 64 contiguous bytes, instead of one 2-byte store per lane per row.
// Rows at or past M and column groups at or past N (N is a multiple of 8)
// are not written; every lane takes part in the shuffles.
template <int kRows>
__device__ __forceinline__ void store_swapped_rows(const float* v, uint16_t* C, int64_t ldc,
                                                   int32_t M, int32_t N, int32_t m0,
                                                   int32_t n_lane, int lane) {
  static_assert(kRows % 8 == 0, "rows come in blocks of eight");
  constexpr int kBlocks = kRows / 8;
  const int j = lane & 7;
  const int32_t n = n_lane - j;  // first of this lane group's eight columns
  float x[kBlocks][8];
#pragma unroll
  for (int b = 0; b < kBlocks; ++b)
#pragma unroll
    for (int k = 0; k < 8; ++k) x[b][k] = v[8 * b + k];
#pragma unroll
  for (int d = 4; d >= 1; d >>= 1) {
    const bool upper = (j & d) != 0;
#pragma unroll
    for (int b = 0; b < kBlocks; ++b) {
#pragma unroll
      for (int k0 = 0; k0 < 8; ++k0) {
        if (k0 & d) continue;
        const int k1 = k0 | d;
        const float out = upper ? x[b][k0] : x[b][k1];
        const float in = __shfl_xor_sync(0xffffffffu, out, d);
        if (upper)
          x[b][k0] = in;
        else
          x[b][k1] = in;
      }
    }
  }
#pragma unroll
  for (int b = 0; b < kBlocks; ++b) {
    const int32_t m = m0 + 8 * b + j;
    if (m < M && n < N)
      ptx::st_global_v4(C + static_cast<size_t>(m) * ldc + n, pack_half2(x[b][0], x[b][1]),
                        pack_half2(x[b][2], x[b][3]), pack_half2(x[b][4], x[b][5]),
                        pack_half2(x[b][6], x[b][7]));
  }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
  constexpr int S = Cfg::kStages;
  constexpr bool kPair = Cfg::kCtas == 2;
  constexpr bool kSplitK = Cfg::kSplit > 1;
  constexpr bool kClustered = Cfg::kClusterCtas > 1;
  // CTA 0's start, for the clock record.
  const bool clk_cta = args.clk != nullptr && blockIdx.x == 0 && threadIdx.x == 0;
  const uint64_t clk_c0 = clk_cta ? clock64() : 0ull;
  const uint64_t clk_t0 = clk_cta ? ptx::globaltimer_ns() : 0ull;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = ptx::smem_addr(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Position of this CTA in its cluster, in its pair, and of the pair in the
  // cluster; units (CTAs, pairs or two-pair clusters) in the grid.
  const uint32_t rank = kClustered ? ptx::cluster_ctarank() : 0u;
  const uint32_t krank = kSplitK ? rank : 0u;  // k-slice of a split-K cluster (0: the leader)
  const uint32_t prank = kPair ? rank : 0u;    // position among the cluster's CTA pairs
  const uint32_t cta = prank & 1u;      // 0: the pair's leader, which issues the MMAs
  const uint32_t pair = prank >> 1;     // which pair of a two-pair cluster
  const uint32_t leader = prank & ~1u;  // cluster rank of this pair's leader
  constexpr uint16_t kClusterMask = static_cast<uint16_t>((1u << Cfg::kClusterCtas) - 1u);
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << leader);
  // Tile column of this pair's tile, from the unit's tile column.
  auto tile_nb = [&](int32_t nbx) { return nbx * Cfg::kMc + static_cast<int32_t>(pair); };
  const int32_t unit = kClustered ? static_cast<int32_t>(ptx::cluster_id_x()) : static_cast<int32_t>(blockIdx.x);
  const int32_t units = kClustered ? static_cast<int32_t>(ptx::num_clusters_x()) : static_cast<int32_t>(gridDim.x);

  const uint32_t bar0 = sb + Cfg::kOffBar;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (S + s); };
  auto bar_tfull = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto bar_tempty = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t bar_mma_done = bar0 + 8u * (2 * S + 4);
  auto bar_tile_full = [&](int i) { return bar0 + 8u * (2 * S + 5 + i); };
  auto bar_tile_empty = [&](int i) { return bar0 + 8u * (2 * S + 7 + i); };
  const uint32_t bar_tile_took = bar0 + 8u * (2 * S + 9);
  const uint32_t bar_red_full = bar0 + 8u * (2 * S + 10);   // split-K: in rank 0
  const uint32_t bar_red_empty = bar0 + 8u * (2 * S + 11);  // split-K: in every rank > 0
  auto sA = [&](int s) { return sb + Cfg::kOffA + s * Cfg::kABytes; };
  auto sB = [&](int s) { return sb + Cfg::kOffB + s * Cfg::kBBytes; };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kOffAbort);
  const Watch w{abort_flag, args.err, args.timeout_ns};
  // Swapped-roles split-K, thread 64: parity + 1 of a red_full phase armed
  // for the other rank's partial and not yet seen complete (0: none).
  uint32_t red_pending = 0;
  // The dynamic tile order as every role reads it (tile_empty lives in the
  // cluster's leader, rank 0, where the scheduler runs).
  const TileRing ring{sb + Cfg::kOffTiles, bar_tile_full(0),
                      kPair ? ptx::mapa(bar_tile_empty(0), 0) : bar_tile_empty(0), w, kPair,
                      warp == 0 && rank == 0 ? bar_tile_took : 0u};
  // Split-K partial tiles in rank 0: slot r - 1 for rank r, element (TMEM
  // lane l, column c) at ((c / 4) * 128 + l) * 16 + (c % 4) * 4 bytes, so a
  // warp's 32 lanes move 512 contiguous bytes per 16-byte access.  (Swapped
  // roles: one slot in every rank, for the half of the columns it finishes.)
  constexpr uint32_t kRedSlotBytes = static_cast<uint32_t>(Cfg::kBM * Cfg::kBN * 4);
  // Epilogue warps of a split-K CTA: rank > 0 writes its accumulator (TMEM
  // buffer at t_row, this thread's lane `lrow`) into its slot of rank 0
  // after rank 0 has emptied the slot, hands the TMEM buffer back and
  // announces the partial with one release arrival per thread.  Returns
  // false if a wait gave up.
  auto splitk_push = [&](uint32_t t_row, int lrow, uint32_t red_par, uint32_t tempty_bar,
                         int32_t tile) -> bool {
    int ok = 1;
    if ((threadIdx.x & 31) == 0)
      ok = wait_bar<true>(bar_red_empty, red_par ^ 1u, w, kSiteRedEmpty, tile) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ptx::named_barrier_and(1, 32 * Cfg::kEpiWarps, ok != 0)) return false;
    const uint32_t dst = ptx::mapa(sb + Cfg::kOffRed + (krank - 1u) * kRedSlotBytes, 0) +
                         static_cast<uint32_t>(lrow) * 16u;
#pragma unroll
    for (int g = 0; g < Cfg::kBN / 16; ++g) {
      uint32_t v[16];
      ptx::tmem_ld_32x32b_x16(t_row + g * 16, v);
      ptx::tmem_wait_ld(v);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ptx::st_shared_cluster_v4(dst + static_cast<uint32_t>((g * 4 + j) * Cfg::kBM) * 16u,
                                  v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
    ptx::tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(tempty_bar);
    ptx::mbar_arrive_release_cluster(ptx::mapa(bar_red_full, 0));
    return true;
  };
  // Rank 0: wait until every other rank's partial of this tile has landed.
  auto splitk_wait_partials = [&](uint32_t red_par, int32_t tile) -> bool {
    int ok = 1;
    if ((threadIdx.x & 31) == 0)
      ok = wait_bar<true>(bar_red_full, red_par, w, kSiteRedFull, tile) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ptx::named_barrier_and(1, 32 * Cfg::kEpiWarps, ok != 0);
  };
  // Rank 0: add the partials' columns [c0, c0 + n) of lane `lrow` to acc, in
  // rank order.
  auto splitk_add = [&](float* acc, int c0, int n, int lrow) {
    for (uint32_t r = 1; r < static_cast<uint32_t>(Cfg::kSplit); ++r) {
      const uint32_t src = sb + Cfg::kOffRed + (r - 1u) * kRedSlotBytes +
                           static_cast<uint32_t>(lrow) * 16u;
#pragma unroll
      for (int g4 = 0; g4 < n / 4; ++g4) {
        const float4 p = ptx::ld_shared_v4_f32(
            src + static_cast<uint32_t>((c0 / 4 + g4) * Cfg::kBM) * 16u);
        acc[4 * g4] += p.x;
        acc[4 * g4 + 1] += p.y;
        acc[4 * g4 + 2] += p.z;
        acc[4 * g4 + 3] += p.w;
      }
    }
  };
  // Rank 0, after reading every partial of the tile: free the slots.
  auto splitk_release_slots = [&]() {
    for (uint32_t r = 1; r < static_cast<uint32_t>(Cfg::kSplit); ++r)
      ptx::mbar_arrive_release_cluster(ptx::mapa(bar_red_empty, r));
  };

  if (threadIdx.x == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmC);
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(bar_full(s), 2);  // the A and B producers of the leader
      ptx::mbar_init(bar_empty(s), Cfg::kPairs);  // one tcgen05.commit per pair of the cluster
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(bar_tfull(b), 1);
      ptx::mbar_init(bar_tempty(b), Cfg::kEpiWarps * Cfg::kCtas);
    }
    ptx::mbar_init(bar_mma_done, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar_tile_full(i), 1);  // the scheduler's publication
      ptx::mbar_init(bar_tile_empty(i), Cfg::kTileConsumers);
    }
    ptx::mbar_init(bar_tile_took, 1);  // the leader's A producer read a tile
    if constexpr (kSplitK) {
      // red_full, plain roles: one arrival per epilogue thread of every rank
      // that sends to rank 0 (each releases its own partial-tile stores);
      // swapped roles: this CTA's own arrival with the expected byte count,
      // which the other rank's asynchronous stores complete.  red_empty: one
      // arrival per epilogue thread of the rank this one sends to (each has
      // read its rows of the slot) -- rank 0 (plain roles) or the other rank
      // (swapped roles).
      ptx::mbar_init(bar_red_full, Cfg::kSwap ? 1 : 32 * Cfg::kEpiWarps * (Cfg::kSplit - 1));
      ptx::mbar_init(bar_red_empty, 32 * Cfg::kEpiWarps);
    }
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc<Cfg::kCtas>(sb + Cfg::kOffSlot, Cfg::kTmemCols);
    ptx::tmem_relinquish<Cfg::kCtas>();
  }
  ptx::tc_fence_before();
  if constexpr (kClustered)
    ptx::cluster_sync();  // every CTA's barriers exist before any uses another's
  else
    __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + Cfg::kOffSlot);
  // Everything above touches only this CTA's shared and tensor memory, so
  // with programmatic dependent launch it overlaps the end of the previous
  // kernel in the stream.  Global memory (A, B, C, the stream-K workspace) is
  // read or written only after that kernel has completed (griddepcontrol.wait
  // in the producer and epilogue roles; the MMA issuer touches none); the
  // next kernel may start its own set-up on SMs as they free up.
  if (warp == 0 || warp == Cfg::kWarpProducerB) {
    {
      // ----------------------------------------------------- TMA producers --
      // One warp per operand: warp 0 loads A, warp kWarpProducerB loads B;
      // the whole warp runs the loop and one elected lane issues the loads.
      const bool is_a = warp == 0;
      const CUtensorMap* tm = is_a ? &tmA : &tmB;
      const bool mn = is_a ? args.a_mn != 0 : args.b_mn != 0;
      // With A multicast this CTA loads one half of its pair's A rows (pair
      // p of the cluster the p-th half) into both pairs' shared memory.
      const bool mc = is_a && Cfg::kMc == 2;
      const int32_t rows = is_a ? Cfg::kBM / Cfg::kMc : Cfg::kBRows;
      const int mn_boxes = rows / 64;
      const uint32_t op_bytes = is_a ? Cfg::kABytes : Cfg::kBBytes;
      const uint32_t op_base = sb + (is_a ? Cfg::kOffA : Cfg::kOffB) +
                               (mc ? pair * (op_bytes / Cfg::kMc) : 0u);
      const uint16_t mc_mask = static_cast<uint16_t>(0x5u << cta);  // this position in both pairs
      // Both CTAs' bytes of this operand are counted on the pair leader's
      // barrier (with multicast: the bytes landing in either CTA of the pair,
      // whichever pair loaded them).
      const uint32_t op_tx = op_bytes * Cfg::kCtas;
      // First row of this CTA's part of the operand in work item `it`: A rows
      // [row, row + rows) or B rows.
      auto row_of = [&](const WorkItem& it) {
        int32_t mb, nbx;
        raster(it.tile, args.tiles_m, args.tiles_n, args.group_m, mb, nbx);
        return is_a ? mb * Cfg::kTileM + static_cast<int32_t>(cta) * Cfg::kBM +
                          static_cast<int32_t>(pair) * rows
                    : tile_nb(nbx) * Cfg::kBN + static_cast<int32_t>(cta) * Cfg::kBRows;
      };
      Sched sched(args, unit, units, ring, static_cast<int32_t>(krank), Cfg::kSplit);
      WorkItem wi;
      // The first work item is worked out before the wait for the previous
      // kernel, so that after it only the loads themselves remain.  So is an
      // L2 prefetch of the item's first k-blocks: it reads nothing into the
      // CTA, and L2 stays coherent with the previous kernel's writes, so the
      // loads after the wait see its results either way; it takes the DRAM
      // latency of the first stages off the kernel's start.
      bool have = sched.next(wi);
      int32_t row = have ? row_of(wi) : 0;
      if (have && ptx::elect_one()) {
        // (With several pairs per cluster, a pair's tile may lie wholly
        // beyond M or N: its loads then only fill zeros, nothing to prefetch.)
        const bool in_range = is_a ? row < args.M : row < args.N;
        const int32_t kb_end = !in_range ? wi.kb0 : wi.kb1 < wi.kb0 + S ? wi.kb1 : wi.kb0 + S;
        for (int32_t kb = wi.kb0; kb < kb_end; ++kb) {
          if (mn) {
            for (int g = 0; g < mn_boxes; ++g)
              ptx::tma_prefetch_l2_2d(tm, row + 64 * g, kb * Cfg::kBK);
          } else {
            ptx::tma_prefetch_l2_2d(tm, kb * Cfg::kBK, row);
          }
        }
      }
      __syncwarp();
      ptx::griddep_wait();
      ptx::griddep_launch_dependents();
      int stage = 0;
      uint32_t phase = 0;
      int64_t fills = 0;
      bool ok = true;
      bool first_item = true;
      for (; ok && have; have = sched.next(wi), row = have ? row_of(wi) : 0) {
        for (int32_t kb = wi.kb0; kb < wi.kb1; ++kb) {
          if (!wait_bar_warp<kPair>(bar_empty(stage), phase ^ 1u, w, kSiteEmpty, wi.tile)) {
            ok = false;
            break;
          }
          const bool skip = args.skip_kb == kb && first_item && unit == 0 && rank == 0;
          if (!skip && ptx::elect_one()) {
            const uint32_t dst = op_base + static_cast<uint32_t>(stage) * op_bytes;
            // K-contiguous: one box of the tile's rows x 64 K-elements.
            // M/N-contiguous: 64 x 64 boxes, 8 KB apart.
            if constexpr (kPair) {
              const uint32_t full_leader = ptx::mapa(bar_full(stage), leader);
              if (cta == 0) ptx::mbar_arrive_expect_tx(bar_full(stage), op_tx);
              if (mc) {
                if (mn) {
                  for (int g = 0; g < mn_boxes; ++g)
                    ptx::tma_load_2d_pair_mc(dst + g * 8192, tm, full_leader, row + 64 * g,
                                             kb * Cfg::kBK, mc_mask);
                } else {
                  ptx::tma_load_2d_pair_mc(dst, tm, full_leader, kb * Cfg::kBK, row, mc_mask);
                }
              } else if (mn) {
                for (int g = 0; g < mn_boxes; ++g)
                  ptx::tma_load_2d_pair(dst + g * 8192, tm, full_leader, row + 64 * g,
                                        kb * Cfg::kBK);
              } else {
                ptx::tma_load_2d_pair(dst, tm, full_leader, kb * Cfg::kBK, row);
              }
            } else {
              ptx::mbar_arrive_expect_tx(bar_full(stage), op_tx);
              if (mn) {
                for (int g = 0; g < mn_boxes; ++g)
                  ptx::tma_load_2d(dst + g * 8192, tm, bar_full(stage), row + 64 * g, kb * Cfg::kBK);
              } else {
                ptx::tma_load_2d(dst, tm, bar_full(stage), kb * Cfg::kBK, row);
              }
            }
          }
          __syncwarp();
          ++fills;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        first_item = false;
      }
      // Drain: the last min(S, fills) fills may still be in use.  Normally
      // wait until the MMA issuer has released each of them, so no tcgen05
      // arrival is still headed for the ring when the CTA exits (tilus "Warp
      // Specialization", "Draining the Pipeline").  When aborting, the CTA
      // holding the full barriers waits instead (bounded, ignoring the abort
      // flag) for those loads to land.
      const int64_t n = fills < S ? fills : S;
      for (int64_t f = fills - n; f < fills; ++f) {
        const int s = static_cast<int>(f % S);
        const uint32_t par = static_cast<uint32_t>((f / S) & 1);
        if (ok) ok = wait_bar_warp<kPair>(bar_empty(s), par, w, kSiteDrain, -1);
        if (!ok && cta == 0)
          wait_bar_warp<kPair>(bar_full(s), par, w, kSiteDrain, -1, /*honor_abort=*/false);
      }
    }
  } else if (warp == 1) {
    if (cta == 0) {
      // ------------------------------------------------------- MMA issuer --
      // The whole warp runs the loop; one elected lane issues every
      // tcgen05.mma and tcgen05.commit.
      const uint32_t idesc = Cfg::kIdesc | (args.a_mn ? ptx::kIdescAMnMajor : 0u) |
                             (args.b_mn ? ptx::kIdescBMnMajor : 0u);
      const uint64_t a_kstep = args.a_mn ? 128u : 2u;
      const uint64_t b_kstep = args.b_mn ? 128u : 2u;
      // Stage 0's descriptors; stage s differs only in the start-address
      // field (address / 16, 14 bits: shared memory stays below 256 KB), so
      // it is stage 0's plus s stages' bytes / 16.  The issue loop is on the
      // tensor pipe's critical path: every instruction saved there counts.
      const uint64_t a_desc0 =
          args.a_mn ? ptx::sw128_mnmajor_desc(sA(0)) : ptx::sw128_kmajor_desc(sA(0));
      const uint64_t b_desc0 =
          args.b_mn ? ptx::sw128_mnmajor_desc(sB(0)) : ptx::sw128_kmajor_desc(sB(0));
      constexpr uint64_t kADescStage = Cfg::kABytes >> 4;
      constexpr uint64_t kBDescStage = Cfg::kBBytes >> 4;
      Sched sched(args, unit, units, ring, static_cast<int32_t>(krank), Cfg::kSplit);
      WorkItem wi;
      int stage = 0;
      uint32_t phase = 0;
      int32_t acc_iter = 0;
      bool ok = true;
      while (ok && sched.next(wi)) {
        const int buf = acc_iter & 1;
        const uint32_t use_par = static_cast<uint32_t>((acc_iter >> 1) & 1);
        if (!wait_bar_warp<kPair>(bar_tempty(buf), use_par ^ 1u, w, kSiteTmemEmpty, wi.tile)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * Cfg::kBN);
        for (int32_t kb = wi.kb0; kb < wi.kb1; ++kb) {
          if (!wait_bar_warp<kPair>(bar_full(stage), phase, w, kSiteFull, wi.tile)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t a_desc = a_desc0 + kADescStage * static_cast<uint32_t>(stage);
          const uint64_t b_desc = b_desc0 + kBDescStage * static_cast<uint32_t>(stage);
          const uint32_t acc_first = kb != wi.kb0 ? 1u : 0u;
          if (ptx::elect_one()) {
#pragma unroll
            for (int k = 0; k < Cfg::kBK / 16; ++k) {
              // One 16-deep K step: +32 bytes inside the swizzled row
              // (K-major) or +16 K-rows = 2048 bytes (MN-major); descriptors
              // count in 16 B.  The first step of the item overwrites the
              // accumulator.  (Steps past K in a last k-block cut by K
              // multiply the zeros the TMA filled in; skipping them measured
              // 2% slower, the issue loop being on the critical path.)
              ptx::mma_f16<Cfg::kCtas>(d_tmem, a_desc + a_kstep * k, b_desc + b_kstep * k, idesc,
                                       k != 0 ? 1u : acc_first);
            }
            // The stage is free once every pair reading it is done: with
            // multicast every pair's issuer releases it in every CTA of the
            // cluster.
            if constexpr (kPair)
              ptx::mma_commit_pair(bar_empty(stage), kClusterMask);
            else
              ptx::mma_commit(bar_empty(stage));
          }
          __syncwarp();
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (ptx::elect_one()) {
          if constexpr (kPair)
            ptx::mma_commit_pair(bar_tfull(buf), pair_mask);
          else
            ptx::mma_commit(bar_tfull(buf));
        }
        __syncwarp();
        ++acc_iter;
      }
      // Every MMA the elected lane issued has finished before tensor memory
      // is freed (bounded, whatever the abort state).
      if (ptx::elect_one()) {
        if constexpr (kPair)
          ptx::mma_commit_pair(bar_mma_done, static_cast<uint16_t>(1u << rank));
        else
          ptx::mma_commit(bar_mma_done);
      }
      __syncwarp();
      wait_bar_warp<kPair>(bar_mma_done, 0u, w, kSiteMmaDone, -1, /*honor_abort=*/false);
    }
  } else if (warp == Cfg::kWarpSched) {
    // ----------------------------------------------------- tile scheduler --
    // Dynamic order: the cluster's leader takes a ticket from the global
    // counter one tile ahead of its A producer (the first ticket at once,
    // each later one when that producer has read the tile before it, i.e.
    // has started it), so tickets go out in the order units start tiles, and
    // publishes the tile (or -1: none left) to the same slot of every CTA of
    // the cluster once that slot is free (all of the cluster's consumer
    // warps have read the slot's last tile).  The last unit to finish sets
    // both counters back to zero for the next launch.
    if (args.tile_ctr != nullptr && rank == 0 && unit < args.dp_tiles) {
      ptx::griddep_wait();  // the counters are global memory
      const int32_t active = units < args.dp_tiles ? units : args.dp_tiles;
      bool ok = true;
      for (int32_t n = 0;; ++n) {
        if (n > 0 && !wait_bar_warp<false>(bar_tile_took, static_cast<uint32_t>((n - 1) & 1), w,
                                           kSiteTileEmpty, -1)) {
          ok = false;
          break;
        }
        uint32_t ticket = 0;
        if (lane == 0) ticket = atomicAdd(args.tile_ctr, 1u);
        ticket = __shfl_sync(0xffffffffu, ticket, 0) + static_cast<uint32_t>(units);
        const int32_t t =
            ticket < static_cast<uint32_t>(args.dp_tiles) ? static_cast<int32_t>(ticket) : -1;
        const int i = n & 1;
        const uint32_t par = static_cast<uint32_t>(((n >> 1) & 1) ^ 1);
        if (!wait_bar_warp<kPair>(bar_tile_empty(i), par, w, kSiteTileEmpty, t)) {
          ok = false;
          break;
        }
        if (lane < Cfg::kClusterCtas) {
          const uint32_t slot = sb + Cfg::kOffTiles + 4u * static_cast<uint32_t>(i);
          if constexpr (kPair) {
            ptx::st_shared_cluster_u32(ptx::mapa(slot, static_cast<uint32_t>(lane)),
                                       static_cast<uint32_t>(t));
            ptx::mbar_arrive_release_cluster(
                ptx::mapa(bar_tile_full(i), static_cast<uint32_t>(lane)));
          } else {
            ptx::st_shared_u32(slot, static_cast<uint32_t>(t));
            ptx::mbar_arrive(bar_tile_full(i));
          }
        }
        __syncwarp();
        if (t < 0) break;
      }
      if (ok && lane == 0) {
        __threadfence();  // this unit's tickets are taken before it counts itself done
        if (atomicAdd(args.tile_ctr + 1, 1u) == static_cast<uint32_t>(active - 1)) {
          args.tile_ctr[0] = 0u;
          args.tile_ctr[1] = 0u;
        }
      }
    }
  } else if constexpr (Cfg::kSwap) {
    // ---------------------------------------------- epilogue, swapped roles --
    ptx::griddep_wait();  // writes C and the workspace
    // The MMA computed a tile of C^T = B x A^T: TMEM lane = column n of C,
    // TMEM column = row m of C.  Each thread owns one column n and holds its
    // kBN values down it; store_swapped_rows turns them around in registers
    // so that each lane writes 8 columns of one row at a time.
    const int q = warp & 3;  // this warp may touch TMEM lanes 32q .. 32q+31 only
    const int row_in_cta = q * 32 + lane;
    const uint32_t tempty_bar0 = bar_tempty(0);
    volatile uint32_t* last_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kOffFlag);
    auto partial = [&](int32_t u, int32_t slot) {
      return args.sk_ws + static_cast<size_t>(u * 2 + slot) * static_cast<size_t>(Cfg::kPartialFloats);
    };
    Sched sched(args, unit, units, ring, static_cast<int32_t>(krank), Cfg::kSplit);
    WorkItem wi;
    int32_t acc_iter = 0;
    // All epilogue warps take the same decision (a failed wait for the next
    // tile ends the loop in every warp, none is left at a barrier below).
    while (ptx::named_barrier_and(1, 32 * Cfg::kEpiWarps, sched.next(wi))) {
      int32_t mb, nb;
      raster(wi.tile, args.tiles_m, args.tiles_n, args.group_m, mb, nb);
      const int buf = acc_iter & 1;
      const uint32_t use_par = static_cast<uint32_t>((acc_iter >> 1) & 1);
      ++acc_iter;
      int ok = 1;
      if (lane == 0) ok = wait_bar<false>(bar_tfull(buf), use_par, w, kSiteTmemFull, wi.tile) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ptx::named_barrier_and(1, 32 * Cfg::kEpiWarps, ok != 0)) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(buf * Cfg::kBN);
      const int32_t n = mb * Cfg::kBM + row_in_cta;  // column of C
      const int32_t m0 = nb * Cfg::kBN;              // first row of C in this tile
      const bool split = !Cfg::kAccF16 && !kSplitK && wi.splits > 1;
      float acc[Cfg::kBN];
      if constexpr (kSplitK) {
        // Rank r finishes rows m0 + r H .. m0 + (r + 1) H - 1 of C
        // (accumulator columns r H .., H = kBN / 2): it sends its partial of
        // the other half to the other rank, keeps its own half and adds the
        // other rank's partial of it.  A sum of two terms: which rank adds
        // does not change the result.  Slot layout as above, for H columns.
        constexpr int kHalf = Cfg::kBN / 2;
        constexpr uint32_t kHalfBytes = static_cast<uint32_t>(Cfg::kBM * kHalf * 4);
        const uint32_t red_par = static_cast<uint32_t>((acc_iter - 1) & 1);
        const uint32_t peer = krank ^ 1u;
        // (a) Arm this CTA's red_full for the other rank's half of this tile
        // (its stores may land before or after), and wait until the other
        // rank has read what this one sent it for the previous tile.
        if (threadIdx.x == 64) {
          ptx::mbar_arrive_expect_tx(bar_red_full, kHalfBytes);
          red_pending = red_par + 1u;
        }
        if (lane == 0)
          ok = wait_bar<true>(bar_red_empty, red_par ^ 1u, w, kSiteRedEmpty, wi.tile) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ptx::named_barrier_and(1, 32 * Cfg::kEpiWarps, ok != 0)) break;
        // (b) Send the other rank's half: asynchronous stores that count
        // themselves on its red_full, so this thread does not wait for them.
        {
          float part[kHalf];
          tmem_ld_f32<kHalf>(t_row + peer * kHalf, part);
          const uint32_t dst =
              ptx::mapa(sb + Cfg::kOffRed, peer) + static_cast<uint32_t>(row_in_cta) * 16u;
          const uint32_t peer_full = ptx::mapa(bar_red_full, peer);
#pragma unroll
          for (int c4 = 0; c4 < kHalf / 4; ++c4)
            ptx::st_async_cluster_v4(dst + static_cast<uint32_t>(c4 * Cfg::kBM) * 16u,
                                     __float_as_uint(part[4 * c4]),
                                     __float_as_uint(part[4 * c4 + 1]),
                                     __float_as_uint(part[4 * c4 + 2]),
                                     __float_as_uint(part[4 * c4 + 3]), peer_full);
        }
        // (c) Own half into registers; the TMEM buffer goes back to the MMA
        // issuer.
        tmem_ld_f32<kHalf>(t_row + krank * kHalf, acc);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(tempty_bar0 + 8u * buf);
        // (d) Add the other rank's partial of this half, free the slot (not
        // after the unit's last tile: nothing more is sent), store.
        if (!splitk_wait_partials(red_par, wi.tile)) break;
        red_pending = 0;
        const uint32_t src = sb + Cfg::kOffRed + static_cast<uint32_t>(row_in_cta) * 16u;
        uint32_t read = 0;  // depends on every value read from the slot
#pragma unroll
        for (int c4 = 0; c4 < kHalf / 4; ++c4) {
          const float4 p = ptx::ld_shared_v4_f32(src + static_cast<uint32_t>(c4 * Cfg::kBM) * 16u);
          acc[4 * c4] += p.x;
          acc[4 * c4 + 1] += p.y;
          acc[4 * c4 + 2] += p.z;
          acc[4 * c4 + 3] += p.w;
          read ^= __float_as_uint(p.x) ^ __float_as_uint(p.y) ^ __float_as_uint(p.z) ^
                  __float_as_uint(p.w);
        }
        if (sched.has_more())
          ptx::mbar_arrive_relaxed_cluster_after(ptx::mapa(bar_red_empty, peer), read);
        store_swapped_rows<kHalf>(acc, args.C, args.ldc, args.M, args.N,
                                  m0 + static_cast<int32_t>(krank) * kHalf, n, lane);
        continue;
      } else if (split) {
        // Same protocol as the plain epilogue: park the fp32 partial, count,
        // and the last contributor sums all partials in unit order.
        float* own = partial(unit, sched.slot_of(unit, wi.sk_tile)) +
                     static_cast<size_t>(row_in_cta) * 4;
#pragma unroll
        for (int g = 0; g < Cfg::kBN / 16; ++g) {
          uint32_t v[16];
          ptx::tmem_ld_32x32b_x16(t_row + g * 16, v);
          ptx::tmem_wait_ld(v);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            ptx::st_global_v4(own + static_cast<size_t>(g * 4 + j) * (Cfg::kBM * 4), v[4 * j],
                              v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(tempty_bar0 + 8u * buf);
        __threadfence();
        ptx::named_barrier_sync(1, 32 * Cfg::kEpiWarps);
        if (threadIdx.x == 64) {
          uint32_t* cnt = args.sk_count + static_cast<size_t>(wi.sk_tile);
          const uint32_t before = atomicAdd(cnt, 1u);
          const bool last = before == static_cast<uint32_t>(wi.splits - 1);
          if (last) *cnt = 0u;
          *last_flag = last ? 1u : 0u;
        }
        ptx::named_barrier_sync(1, 32 * Cfg::kEpiWarps);
        if (*last_flag == 0u) continue;
        __threadfence();
#pragma unroll
        for (int i = 0; i < Cfg::kBN; ++i) acc[i] = 0.0f;
        for (int32_t j = 0; j < wi.splits; ++j) {
          const int32_t u = wi.first_unit + j;
          const float* src = partial(u, sched.slot_of(u, wi.sk_tile)) +
                             static_cast<size_t>(row_in_cta) * 4;
#pragma unroll
          for (int g4 = 0; g4 < Cfg::kBN / 4; ++g4) {
            const float4 v = ptx::ld_global_cg_v4(src + static_cast<size_t>(g4) * (Cfg::kBM * 4));
            acc[4 * g4] += v.x;
            acc[4 * g4 + 1] += v.y;
            acc[4 * g4 + 2] += v.z;
            acc[4 * g4 + 3] += v.w;
          }
        }
      } else {
#pragma unroll
        for (int g = 0; g < Cfg::kBN / 16; ++g) {
          if constexpr (Cfg::kAccF16) {
            uint32_t v[8];
            ptx::tmem_ld_32x32b_x8_pack16(t_row + g * 16, v);
            ptx::tmem_wait_ld(v);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const __half2 h = *reinterpret_cast<const __half2*>(&v[i]);
              acc[g * 16 + 2 * i] = __low2float(h);
              acc[g * 16 + 2 * i + 1] = __high2float(h);
            }
          } else {
            uint32_t v[16];
            ptx::tmem_ld_32x32b_x16(t_row + g * 16, v);
            ptx::tmem_wait_ld(v);
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[g * 16 + i] = __uint_as_float(v[i]);
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(tempty_bar0 + 8u * buf);
      }
      store_swapped_rows<Cfg::kBN>(acc, args.C, args.ldc, args.M, args.N, m0, n, lane);
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    ptx::griddep_wait();  // writes C and the workspace
    const int q = warp & 3;  // this warp may touch TMEM lanes 32q .. 32q+31 only
    const int row_in_cta = q * 32 + lane;
    const uint32_t stage_base = sb + Cfg::kOffEpi + static_cast<uint32_t>(q * 2 * Cfg::kEpiBufBytes);
    // tmem_empty lives in the leader CTA: every epilogue warp of the pair
    // arrives there.
    const uint32_t tempty_bar0 = kPair ? ptx::mapa(bar_tempty(0), leader) : bar_tempty(0);
    volatile uint32_t* last_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kOffFlag);
    // This CTA's share of unit u's partial tile in slot `slot`.
    auto partial = [&](int32_t u, int32_t slot) {
      return args.sk_ws + (static_cast<size_t>(u * 2 + slot) * Cfg::kClusterCtas + rank) *
                              static_cast<size_t>(Cfg::kPartialFloats);
    };
    Sched sched(args, unit, units, ring, static_cast<int32_t>(krank), Cfg::kSplit);
    WorkItem wi;
    uint32_t stores = 0;
    int32_t acc_iter = 0;
    // All epilogue warps take the same decision (a failed wait for the next
    // tile ends the loop in every warp, none is left at a barrier below).
    while (ptx::named_barrier_and(1, 32 * Cfg::kEpiWarps, sched.next(wi))) {
      int32_t mb, nbx;
      raster(wi.tile, args.tiles_m, args.tiles_n, args.group_m, mb, nbx);
      const int32_t nb = tile_nb(nbx);
      const int buf = acc_iter & 1;
      const uint32_t use_par = static_cast<uint32_t>((acc_iter >> 1) & 1);
      ++acc_iter;
      int ok = 1;
      if (lane == 0) ok = wait_bar<kPair>(bar_tfull(buf), use_par, w, kSiteTmemFull, wi.tile) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // All epilogue warps take the same decision, so none is left waiting at
      // a barrier below for a warp that gave up.
      if (!ptx::named_barrier_and(1, 32 * Cfg::kEpiWarps, ok != 0)) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(buf * Cfg::kBN);
      const int32_t row0 = mb * Cfg::kTileM + static_cast<int32_t>(cta) * Cfg::kBM + q * 32;
      const bool split = !Cfg::kAccF16 && !kSplitK && wi.splits > 1;
      const uint32_t red_par = static_cast<uint32_t>((acc_iter - 1) & 1);
      if constexpr (kSplitK) {
        if (krank != 0) {
          if (!splitk_push(t_row, row_in_cta, red_par, tempty_bar0 + 8u * buf, wi.tile)) break;
          continue;  // rank 0 stores the tile
        }
        if (!splitk_wait_partials(red_par, wi.tile)) break;
      }
      if (split) {
        // Stream-K tail tile shared with other units.  (a) Park this unit's
        // partial accumulator (fp32) in its workspace slot and give the TMEM
        // buffer back.
        // Partial tile layout [column / 4][row][column % 4]: for a fixed group
        // of four columns the warp's 32 rows are 512 contiguous bytes, so every
        // store (and the fix-up's loads) is one fully used burst.
        float* own = partial(unit, sched.slot_of(unit, wi.sk_tile)) +
                     static_cast<size_t>(row_in_cta) * 4;
#pragma unroll 1
        for (int c = 0; c < Cfg::kBN / 32; ++c) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c * 32, v);
          ptx::tmem_wait_ld(v);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            ptx::st_global_v4(own + static_cast<size_t>(c * 8 + j) * (Cfg::kBM * 4), v[4 * j],
                              v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kPair)
            ptx::mbar_arrive_cluster(tempty_bar0 + 8u * buf);
          else
            ptx::mbar_arrive(tempty_bar0 + 8u * buf);
        }
        // (b) Count this contribution.  Whoever brings the count to `splits`
        // holds the last piece: it resets the counter for the next launch and
        // finishes the tile.  Nobody waits for anybody.
        __threadfence();
        ptx::named_barrier_sync(1, 32 * Cfg::kEpiWarps);
        if (threadIdx.x == 64) {
          uint32_t* cnt = args.sk_count + static_cast<size_t>(wi.sk_tile) * Cfg::kClusterCtas + rank;
          const uint32_t before = atomicAdd(cnt, 1u);
          const bool last = before == static_cast<uint32_t>(wi.splits - 1);
          if (last) *cnt = 0u;
          *last_flag = last ? 1u : 0u;
        }
        ptx::named_barrier_sync(1, 32 * Cfg::kEpiWarps);
        if (*last_flag == 0u) continue;
        __threadfence();
      }
      // Stage one 32 x 64 chunk of fp16 C through this warp's swizzled
      // shared-memory buffers and store it with the TMA engine.
      auto store_chunk = [&](const uint32_t (&packed)[32], int c) {
        const uint32_t sbuf = stage_base + (stores & 1u) * Cfg::kEpiBufBytes;
        if (stores >= 2 && lane == 0) ptx::bulk_wait_group_read<1>();
        __syncwarp();
        // Row `lane` of the 32x64 staging tile, 16-byte chunk j stored at
        // chunk position j ^ (row % 8): the 128-byte swizzle the C tensor
        // map expects, and conflict-free across the warp.
        const uint32_t row_addr = sbuf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          ptx::st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4),
                            packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        const int32_t col0 = nb * Cfg::kBN + c * 64;
        if (lane == 0 && row0 < args.M && col0 < args.N) {
          ptx::tma_store_2d(&tmC, sbuf, col0, row0);
          ptx::bulk_commit_group();
          ++stores;
        }
        stores = __shfl_sync(0xffffffffu, stores, 0);
      };
      // The whole accumulator buffer is in registers: hand it back.
      auto release_tmem = [&]() {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kPair)
            ptx::mbar_arrive_cluster(tempty_bar0 + 8u * buf);
          else
            ptx::mbar_arrive(tempty_bar0 + 8u * buf);
        }
      };
      if constexpr (kSplitK) {
        // Rank 0: its own accumulator plus the other ranks' partials, in
        // rank order.
#pragma unroll 1
        for (int c = 0; c < Cfg::kBN / 64; ++c) {
          uint32_t v0[32], v1[32];
          ptx::tmem_ld_32x32b_x32(t_row + c * 64, v0);
          ptx::tmem_ld_32x32b_x32(t_row + c * 64 + 32, v1);
          ptx::tmem_wait_ld(v0);
          ptx::tmem_regs_ready(v1);
          float acc[64];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            acc[i] = __uint_as_float(v0[i]);
            acc[32 + i] = __uint_as_float(v1[i]);
          }
          if (c == Cfg::kBN / 64 - 1) release_tmem();
          splitk_add(acc, c * 64, 64, row_in_cta);
          // Nothing more is sent after the unit's last tile.
          if (c == Cfg::kBN / 64 - 1 && sched.has_more()) splitk_release_slots();
          uint32_t packed[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) packed[i] = pack_half2(acc[2 * i], acc[2 * i + 1]);
          store_chunk(packed, c);
        }
      } else if (split) {
#pragma unroll 1
        for (int c = 0; c < Cfg::kBN / 64; ++c) {
          // (c) The tile's value: the contributors' partials summed in unit
          // order, so the result does not depend on who finished last.
          float acc[64];
#pragma unroll
          for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
          for (int32_t j = 0; j < wi.splits; ++j) {
            const int32_t u = wi.first_unit + j;
            const float* src = partial(u, sched.slot_of(u, wi.sk_tile)) +
                               static_cast<size_t>(row_in_cta) * 4 +
                               static_cast<size_t>(c * 16) * (Cfg::kBM * 4);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float4 v = ptx::ld_global_cg_v4(src + static_cast<size_t>(i) * (Cfg::kBM * 4));
              acc[4 * i] += v.x;
              acc[4 * i + 1] += v.y;
              acc[4 * i + 2] += v.z;
              acc[4 * i + 3] += v.w;
            }
          }
          uint32_t packed[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) packed[i] = pack_half2(acc[2 * i], acc[2 * i + 1]);
          store_chunk(packed, c);
        }
      } else if constexpr (Cfg::kAccF16) {
#pragma unroll 1
        for (int c = 0; c < Cfg::kBN / 64; ++c) {
          uint32_t packed[32];
          ptx::tmem_ld_32x32b_x32_pack16(t_row + c * 64, packed);
          ptx::tmem_wait_ld(packed);
          if (c == Cfg::kBN / 64 - 1) release_tmem();
          store_chunk(packed, c);
        }
      } else {
        // fp32 accumulator: the TMEM loads of chunk c + 1 are issued as soon
        // as chunk c is packed, so they run while chunk c is staged and
        // stored.
        uint32_t v0[32], v1[32];
        ptx::tmem_ld_32x32b_x32(t_row, v0);
        ptx::tmem_ld_32x32b_x32(t_row + 32, v1);
#pragma unroll 1
        for (int c = 0; c < Cfg::kBN / 64; ++c) {
          uint32_t packed[32];
          ptx::tmem_wait_ld(v0);
          ptx::tmem_regs_ready(v1);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            packed[i] = pack_half2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
            packed[16 + i] = pack_half2(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1]));
          }
          ptx::tmem_regs_ready(packed);  // packed before v0 and v1 are loaded again
          if (c + 1 < Cfg::kBN / 64) {
            ptx::tmem_ld_32x32b_x32(t_row + (c + 1) * 64, v0);
            ptx::tmem_ld_32x32b_x32(t_row + (c + 1) * 64 + 32, v1);
          } else {
            release_tmem();
          }
          store_chunk(packed, c);
        }
      }
    }
    if (lane == 0) ptx::bulk_wait_group<0>();
    __syncwarp();
  }

  ptx::tc_fence_before();
  if constexpr (kSplitK) {
    // No CTA leaves while another may still touch its memory.  In a split-K
    // cluster every such access (a partial tile, an arrival on red_full or
    // red_empty) is waited for by the CTA it targets before that CTA gets
    // here, unless a wait gave up: then a swapped-roles CTA first waits
    // (bounded) for the partial it armed red_full for, and the cluster
    // barrier releases and acquires.  Otherwise it need not order memory;
    // a release arrival would wait for this thread's stores of C to
    // complete (~0.45 us at the end of every launch).
    if (threadIdx.x == 64 && red_pending != 0u && *abort_flag != 0u)
      wait_bar<true>(bar_red_full, red_pending - 1u, w, kSiteRedFull, -1, false);
    __syncthreads();  // after it every thread reads the same abort flag
    if (*abort_flag != 0u)
      ptx::cluster_sync();
    else
      ptx::cluster_sync_relaxed();
  } else if constexpr (kClustered) {
    ptx::cluster_sync();  // no CTA leaves while another may still touch its memory
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<Cfg::kCtas>(tmem_base, Cfg::kTmemCols);
  }
  if (clk_cta) {
    const uint64_t c1 = clock64();
    const uint64_t t1 = ptx::globaltimer_ns();
    atomicAdd(args.clk, 1ull);
    atomicAdd(args.clk + 1, static_cast<unsigned long long>(c1 - clk_c0));
    atomicAdd(args.clk + 2, static_cast<unsigned long long>(t1 - clk_t0));
  }
}

// C := 0 for K == 0 (the empty sum).  C rows are a multiple of 16 bytes.
__global__ void gemm_zero_fill(uint4* c, int64_t n16) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    c[i] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace gb300
