// gemm.cu -- host side of the C ABI declared in include/gemm.h: argument
// checks, plans, tensor-map encoding and kernel launch for the sm_103a GEMM
// C = A x B^T (tilus "A Minimal Hopper Matmul", section "Block Tiling").
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <utility>

#include "gemm.h"
#include "gemm_kernel.cuh"

#define GB300_GEMM_VERSION "0.1.0"

namespace {

using gb300::GemmArgs;
using gb300::GemmCfg;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// ------------------------------------------------------------ the variants --
// Compile-time tile configurations; the host picks one per call.
using PairF32 = GemmCfg<2, 6, false>;    // CTA pair, 256 x 256 tile, 6 stages
using PairF16 = GemmCfg<2, 6, true>;
using SingleF32 = GemmCfg<1, 4, false>;  // one CTA, 128 x 256 tile, 4 stages
using SingleF16 = GemmCfg<1, 4, true>;
using Pair128F32 = GemmCfg<2, 8, false, 128>;   // CTA pair, 256 x 128 tile, 8 stages
using Pair128F16 = GemmCfg<2, 8, true, 128>;
using Single64F32 = GemmCfg<1, 8, false, 64>;   // one CTA, 128 x 64 tile, 8 stages
using Single64F16 = GemmCfg<1, 8, true, 64>;
// Swapped roles for small M: 128 columns of C x 16/32/64 rows of C per CTA.
using Swap16F32 = GemmCfg<1, 11, false, 16, true>;
using Swap16F16 = GemmCfg<1, 11, true, 16, true>;
using Swap32F32 = GemmCfg<1, 10, false, 32, true>;
using Swap32F16 = GemmCfg<1, 10, true, 32, true>;
using Swap64F32 = GemmCfg<1, 8, false, 64, true>;
using Swap64F16 = GemmCfg<1, 8, true, 64, true>;
// Two CTA pairs per cluster sharing the A block of their tile-row (multicast).
using PairMcF32 = GemmCfg<2, 6, false, 256, false, 2>;
using PairMcF16 = GemmCfg<2, 6, true, 256, false, 2>;
// Split-K clusters (fp32 accumulation only): the CTAs of a cluster share each
// tile, one k-slice each, and add their partials through shared memory.
using Swap16K2F32 = GemmCfg<1, 11, false, 16, true, 1, 2>;
using Swap32K2F32 = GemmCfg<1, 10, false, 32, true, 1, 2>;
using Swap64K2F32 = GemmCfg<1, 8, false, 64, true, 1, 2>;
using Single64K4F32 = GemmCfg<1, 4, false, 64, false, 1, 4>;

struct VariantInfo {
  const char* name;
  int ctas;            // CTAs per unit (cluster size)
  int tile_m, tile_n;  // output tile (rows x columns of C) owned by one unit: a CTA, a CTA
                       // pair, or two pairs side by side in N
  int box_a_rows;      // rows of A each CTA loads per stage (K-contiguous A)
  int box_b_rows;      // rows of B each CTA loads per stage
  bool swap;           // MMA roles swapped: the kernel's tiles run over (N, M)
  int ksplit;          // CTAs of a split-K cluster sharing each tile (1: none)
  int base;            // the variant with whole tiles per CTA it refines (itself if none)
};

constexpr int kVariantPair = 0;
constexpr int kVariantSingle = 1;
constexpr int kVariantPair128 = 2;
constexpr int kVariantSingle64 = 3;
constexpr int kVariantSwap16 = 4;
constexpr int kVariantSwap32 = 5;
constexpr int kVariantSwap64 = 6;
constexpr int kVariantPairMc = 7;
constexpr int kVariantSwap16K2 = 8;
constexpr int kVariantSwap32K2 = 9;
constexpr int kVariantSwap64K2 = 10;
constexpr int kVariantSingle64K4 = 11;
constexpr int kNumVariants = 12;
constexpr VariantInfo kVariants[kNumVariants] = {
    {"tc_pair_256x256_s6", 2, 256, 256, 128, 128, false, 1, 0},
    {"tc_single_128x256_s4", 1, 128, 256, 128, 256, false, 1, 1},
    {"tc_pair_256x128_s8", 2, 256, 128, 128, 64, false, 1, 2},
    {"tc_single_128x64_s8", 1, 128, 64, 128, 64, false, 1, 3},
    {"tc_swap_16x128_s11", 1, 16, 128, 16, 128, true, 1, 4},
    {"tc_swap_32x128_s10", 1, 32, 128, 32, 128, true, 1, 5},
    {"tc_swap_64x128_s8", 1, 64, 128, 64, 128, true, 1, 6},
    {"tc_pair_mc_256x256_s6", 4, 256, 512, 64, 128, false, 1, 7},
    {"tc_swap_16x128_k2", 2, 16, 128, 16, 128, true, 2, kVariantSwap16},
    {"tc_swap_32x128_k2", 2, 32, 128, 32, 128, true, 2, kVariantSwap32},
    {"tc_swap_64x128_k2", 2, 64, 128, 64, 128, true, 2, kVariantSwap64},
    {"tc_single_128x64_k4", 4, 128, 64, 128, 64, false, 4, kVariantSingle64},
};

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s for any single wait
constexpr size_t kRecordBytes = 64;  // watchdog record (16 B) + clock record (3 x 8 B)
constexpr int kGroupM = 8;                             // raster group height, tiles
// Tensor-map cache: kMapSets sets of kMapWays entries (1024 maps, ~200 KB per
// plan), so that a caller cycling through a few hundred operand buffers
// (three maps per call) still finds every map it made.
constexpr int kMapSets = 128;
constexpr int kMapWays = 8;
// gemm_run_host's pipeline: at most kHostChunksA row chunks of A and
// kHostChunksB of B, and at most kHostBlocks blocks of C.
constexpr int kHostChunksA = 32;
constexpr int kHostChunksB = 8;
constexpr int kHostBlocks = 64;

struct MapEntry {
  const void* ptr;
  uint64_t rows, cols, pitch;
  uint32_t box_rows, box_cols;
  uint64_t stamp;
  CUtensorMap map;
};

}  // namespace

struct gemm_plan_s {
  int device = 0;
  int num_sms = 0;
  int max_pairs = 0;  // CTA pairs of the pair kernel that fit on the device at once
  int max_quads = 0;  // two-pair clusters of the multicast kernel that fit at once
  int max_units[kNumVariants] = {};  // units (CTAs or clusters) of each variant that fit at once
  // Stream-K workspace, allocated once at plan creation: partial fp32 tiles
  // (2 slots per unit) and per-tile contribution counters (kept at zero
  // between launches by the kernel itself).
  float* sk_ws = nullptr;
  uint32_t* sk_count = nullptr;
  size_t sk_count_words = 0;
  // Dynamic tile order: ticket and finished-unit counters (two words after
  // the stream-K counters, kept at zero between launches by the kernel).
  uint32_t* tile_ctr = nullptr;
  int32_t tile_order = 0;  // 0 automatic, 1 static round robin, 2 dynamic when possible
  int32_t schedule_mode = 0;  // 0 auto, 1 whole tiles only, 2 stream-K tail whenever possible
  EncodeTiledFn encode = nullptr;
  uint32_t* d_err = nullptr;  // 4-word watchdog record, then the clock record
  unsigned long long* d_clk = nullptr;  // [launches, SM cycles, ns] of CTA 0 (inside d_err's block)
  uint32_t last_err[4] = {0, 0, 0, 0};
  uint64_t timeout_ns = kDefaultTimeoutNs;
  int32_t skip_kb = -1;
  int32_t forced_variant = -1;
  bool pdl = true;  // programmatic dependent launch of the GEMM kernel
  bool clock_record = false;  // kernels add to the clock record (gemm_plan_set_clock_record)
  uint64_t launches = 0;
  uint64_t clock = 0;
  MapEntry maps[kMapSets][kMapWays];
  // device staging for gemm_run_host
  void* dA = nullptr;
  void* dB = nullptr;
  void* dC = nullptr;
  size_t capA = 0, capB = 0, capC = 0;
  // gemm_run_host's copy-in, compute and copy-out streams and their events
  // (created on first use): one per input chunk, one per block of C.
  cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
  cudaEvent_t ev_start = nullptr;
  cudaEvent_t ev_in[kHostChunksA + kHostChunksB] = {};
  cudaEvent_t ev_comp[kHostBlocks] = {};
};

namespace {

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// L2 promotion of the operand loads.  Rows whose pitch is not a multiple of
// 128 bytes straddle L2 lines; there promoting each request to 256 bytes
// costs more than it saves (measured ~6% slower at K = 4104), so promote by
// 128 bytes.
CUtensorMapL2promotion l2_promotion(uint64_t pitch_bytes) {
  return pitch_bytes % 128 == 0 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
}

// True if `ptr` lies in memory allocated on device `dev` (cudaMalloc,
// cudaMallocAsync, or virtual memory mapped there).  Host, managed and
// unregistered memory, and another GPU's memory, are refused: the kernel's
// tensor maps must cover this GPU's own memory.
bool on_device(const void* ptr, int dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice && at.device == dev;
}

enum MapResult { kMapOk = 0, kMapNotDevice = 1, kMapEncodeFailed = 2 };

// Tensor map of a row-major fp16 [rows, cols] whose rows are `pitch`
// elements apart (0: cols), from the plan's cache.  A pointer is checked to be
// memory of the plan's device when its map is made (a cache miss): a cached
// map stands for a pointer already checked.
MapResult get_map(gemm_plan_s* p, CUtensorMap* out, const void* ptr, uint64_t rows,
                  uint64_t cols, uint32_t box_rows, uint32_t box_cols, uint64_t pitch = 0) {
  if (pitch == 0) pitch = cols;
  // The set: a mix of the key's fields (an address, its shape and box).
  uint64_t h = reinterpret_cast<uintptr_t>(ptr) >> 8;
  h ^= rows * 0x9e3779b97f4a7c15ull ^ cols * 0xc2b2ae3d27d4eb4full ^ pitch * 0x165667b19e3779f9ull ^
       (static_cast<uint64_t>(box_rows) << 32 | box_cols) * 0xd6e8feb86659fd93ull;
  h ^= h >> 29;
  MapEntry* set = p->maps[(h * 0xbf58476d1ce4e5b9ull >> 40) % kMapSets];
  MapEntry* victim = &set[0];
  for (int i = 0; i < kMapWays; ++i) {
    MapEntry& e = set[i];
    if (e.stamp && e.ptr == ptr && e.rows == rows && e.cols == cols && e.pitch == pitch &&
        e.box_rows == box_rows && e.box_cols == box_cols) {
      e.stamp = ++p->clock;
      *out = e.map;
      return kMapOk;
    }
    if (e.stamp < victim->stamp) victim = &e;
  }
  if (!on_device(ptr, p->device)) return kMapNotDevice;
  // Row-major fp16 [rows, cols]: dimension 0 is the contiguous one.
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = p->encode(&victim->map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr),
                         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, l2_promotion(pitch * 2),
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    victim->stamp = 0;
    return kMapEncodeFailed;
  }
  victim->ptr = ptr;
  victim->rows = rows;
  victim->cols = cols;
  victim->pitch = pitch;
  victim->box_rows = box_rows;
  victim->box_cols = box_cols;
  victim->stamp = ++p->clock;
  *out = victim->map;
  return kMapOk;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Shape and enum checks shared by gemm_run and gemm_run_host.
gemm_status_t check_shape(int64_t M, int64_t N, int64_t K, gemm_acc_t acc) {
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_INVALID_ARG;
  if (acc != GEMM_ACC_F32 && acc != GEMM_ACC_F16) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (K % 8 != 0 || N % 8 != 0) return GEMM_ERR_ALIGNMENT;
  return GEMM_OK;
}

int64_t tiles_of(const VariantInfo& vi, int64_t M, int64_t N) {
  return ((M + vi.tile_m - 1) / vi.tile_m) * ((N + vi.tile_n - 1) / vi.tile_n);
}

constexpr int64_t kMinSkIters = 16;  // fewest k-blocks a stream-K unit is given
constexpr double kSkFixupKb = 2.0;   // cost of a partial-tile fix-up, in k-block times
constexpr double kSkMinGain = 0.97;  // use the stream-K tail only if it saves >= 3%

// How one call is laid out on the device.
struct Schedule {
  int variant;
  int64_t units;      // CTAs or CTA pairs launched
  int grid;           // CTAs launched
  int64_t dp_tiles;   // tiles handed out whole
  int64_t sk_units;   // units sharing the stream-K tail (0 = none)
  int64_t sk_iters;   // k-blocks in the tail
  bool dyn;           // whole tiles after each unit's first come in the dynamic order
};

// Whole tiles are dealt round robin to U persistent units (U = CTA pairs or
// CTAs that fit at once).  When T tiles are not a multiple of U the last wave
// runs part-empty; then its T % U tiles become a stream-K share whose
// k-blocks are split evenly over the units (each unit runs its share before
// its whole tiles), if the estimate (in k-block times per unit) says it saves
// enough.  The testing mode 2 forces the share on any shape.
// Automatic choice, from measurements on GB300 (N = K = 8192 unless noted):
// swapped roles when C has at most 64 rows (the tile then wastes no MMA rows
// on padding and the work is spread over all SMs: 16 rows 32 us vs 42 us);
// one CTA with 128 x 64 tiles up to 128 rows (more, narrower tiles: 41 us vs
// 46 us for the pair); the CTA-pair kernel above that.
// Very small problems (fewer 256 x 256 tiles than a quarter of the resident
// pairs) also go to the 128 x 64 tiles, which spread their few k-blocks over
// more SMs (512^3: 11.1 us vs 13.2 us; 1024^3: 11.2 us vs 13.4 us).
// K-contiguous rows whose pitch is not a multiple of 128 bytes (K % 64 != 0)
// make every 128-byte TMA row straddle two L2 lines, doubling the load
// requests each SM issues; there two pairs share A by multicast, halving A's
// requests (3000 x 5000 x 4104: 1514 vs 1311 TFLOP/s).  On aligned rows it
// ties with the one-pair kernel when the clock is not capped (8192^3: 1884 vs
// 1871) and lost 6% once power-capped, with 144 of the 152 SMs in use.
int auto_variant(int64_t M, int64_t N, int64_t K, bool k_major, int max_pairs, int max_quads) {
  if (M <= 16) return kVariantSwap16;
  if (M <= 32) return kVariantSwap32;
  if (M <= 64) return kVariantSwap64;
  if (M <= 128) return kVariantSingle64;
  const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
  if (4 * pair_tiles < max_pairs) return kVariantSingle64;
  if (k_major && K % 64 != 0 && max_quads > 0) return kVariantPairMc;
  return kVariantPair;
}

// The split-K cluster variant to use instead of variant v for T tiles of KB
// k-blocks, or -1.  With swapped roles, when every tile would be cut into
// exactly two k-pieces (T <= U / 2), a cluster of two CTAs per tile adds the
// second piece's partial through shared memory, instead of parking both in
// global memory and counting them (64 x 8192^2 +8%, 16 and 32 x 8192^2 +7%,
// alternating runs on GB300).  A problem of few 128 x 64 tiles (T at most a
// quarter of the SMs) with at least 8 k-blocks per CTA takes four CTAs per
// tile, so that each CTA loads a quarter of the tile's operands
// (128 x 1024 x 8192 2.4x, 256 x 256 x 4096 1.8x); with fewer (512^3: 2 per
// CTA) launching the four-CTA clusters costs more than it saves (-22%).
int split_k_variant(int v, int64_t T, int64_t KB, const int* max_units) {
  int ks = -1;
  if (kVariants[v].swap && kVariants[v].ksplit == 1) {
    const int64_t U = max_units[v];
    const int64_t pieces = T > 0 ? std::min<int64_t>(U / T, KB / kMinSkIters) : 0;
    const bool cut = T < U && (kVariants[v].tile_m >= 32 || 2 * T <= U);
    if (cut && pieces == 2)
      ks = v == kVariantSwap16 ? kVariantSwap16K2 : v == kVariantSwap32 ? kVariantSwap32K2
                                                                         : kVariantSwap64K2;
  } else if (v == kVariantSingle64) {
    if (4 * T <= max_units[kVariantSingle64] && KB >= 4 * 8) ks = kVariantSingle64K4;
  }
  if (ks >= 0 && (T > max_units[ks] || KB < kVariants[ks].ksplit)) ks = -1;
  return ks;
}

// `mn`: an operand is stored M- or N-contiguous (the swapped-roles variants
// take K-contiguous operands only).
Schedule make_schedule(const gemm_plan_s* p, int64_t M, int64_t N, int64_t K, gemm_acc_t acc,
                       bool mn = false) {
  int v = p->forced_variant >= 0 ? p->forced_variant
                                 : auto_variant(M, N, K, !mn, p->max_pairs, p->max_quads);
  if (mn && kVariants[v].swap) v = M <= 128 ? kVariantSingle64 : kVariantPair;
  const int64_t KB = (K + 63) / 64;
  // Split-K clusters take fp32 accumulation and at least one k-block per CTA.
  if (kVariants[v].ksplit > 1 && (acc != GEMM_ACC_F32 || KB < kVariants[v].ksplit))
    v = kVariants[v].base;
  if (kVariants[v].ctas == 4 && p->max_quads < 1) v = kVariantPair;
  if (kVariants[v].ctas == 2 && p->max_pairs < 1) v = kVariantSingle;
  if (p->max_units[v] < 1) v = kVariants[v].base;
  // Automatic choice of a split-K cluster: few tiles, each with many
  // k-blocks, spread over the SMs by cutting K instead of sharing partial
  // tiles through global memory (see split_k_variant).
  if (p->forced_variant < 0 && p->schedule_mode == 0 && acc == GEMM_ACC_F32) {
    const int ks = split_k_variant(v, tiles_of(kVariants[v], M, N), KB, p->max_units);
    if (ks >= 0) v = ks;
  }
  const VariantInfo& vi = kVariants[v];
  const int64_t T = tiles_of(vi, M, N);
  const int64_t U = p->max_units[v];
  Schedule s;
  s.variant = v;
  s.units = T < U ? T : U;
  s.dp_tiles = T;
  s.sk_units = 0;
  s.sk_iters = 0;
  s.dyn = false;
  // The share pays only when whole tiles follow it (T >= U): the partial-tile
  // fix-ups then overlap those tiles' main loops.  With nothing after it, the
  // fix-ups end the kernel and cost more than the part-empty wave they save.
  // With swapped roles a partial tile is small (128 x 16..64 fp32), so the
  // share is cheap even with no whole tiles after it: it is what spreads a
  // few tall tiles over every SM.
  const bool allowed = acc == GEMM_ACC_F32 && p->sk_ws && p->sk_count && KB > 0 &&
                       p->schedule_mode != 1 && vi.ksplit == 1 &&
                       ((T % U != 0 && (T >= U || vi.swap)) || p->schedule_mode == 2);
  if (allowed) {
    // Only the tiles of the part-empty last wave are shared (all tiles when
    // T < U): the smaller the share, the more of the work runs as whole tiles,
    // whose concurrent units load the same k-blocks and share them in L2.
    // Measured against sharing T % U + U tiles: 4096 x 4096 x 1024 +26%,
    // 2048 x 8192 x 8192 +7%, 3000 x 5000 x 4104 +1.6%, 8192^3 unchanged.
    const int64_t sk_tiles = T >= U ? (T % U != 0 ? T % U : U) : T;
    const int64_t dp = T - sk_tiles;
    const int64_t iters = sk_tiles * KB;
    // Forced mode (testing) lets units take as little as one k-block, so
    // tiles get many contributors.
    int64_t usk = iters / (p->schedule_mode == 2 ? 1 : kMinSkIters);
    if (usk > U) usk = U;
    // At most about four contributors per tile: the last one reads the
    // others' partial tiles, and that read grows with their number.
    if (p->schedule_mode != 2 && !vi.swap && usk > 4 * sk_tiles) usk = 4 * sk_tiles;
    // Swapped roles with fewer tall tiles than units: the fix-up of a tile
    // shared by units whose ranges cross tile ends is the launch's tail, so
    // cut every tile into the same whole number of pieces (T x floor(U / T)
    // units; one piece = whole tiles on T units) when the partial tiles are
    // large (32 or 64 rows of C) or there are pieces to spare (2T <= U):
    // 64 x 8192^2 +8%, 48 x 12288 x 8192 +11%, 16 x 8192^2 +2%; with 16 rows
    // and 128 tiles the units' continuous ranges are faster (16 x 16384^2:
    // 97 vs 92 TFLOP/s).
    // Every unit keeps at least kMinSkIters k-blocks (the fix-up counts on
    // every unit of the share contributing).
    if (p->schedule_mode == 0 && vi.swap && T < U && (vi.tile_m >= 32 || 2 * T <= U)) {
      const int64_t pieces = std::min<int64_t>(U / T, KB / kMinSkIters);
      usk = pieces > 1 ? T * pieces : 0;  // one piece per tile: whole tiles, no share
    }
    const bool fits = static_cast<size_t>(sk_tiles * vi.ctas) <= p->sk_count_words;
    if (usk >= 2 && fits) {
      const double t_dp = static_cast<double>((T + U - 1) / U) * KB;
      const double t_sk = static_cast<double>(dp / U) * KB +
                          static_cast<double>((iters + usk - 1) / usk) + kSkFixupKb;
      if (p->schedule_mode == 2 || t_sk < kSkMinGain * t_dp) {
        s.units = dp > 0 ? U : usk;
        s.dp_tiles = dp;
        s.sk_units = usk;
        s.sk_iters = iters;
      }
    }
  }
  // Dynamic order of whole tiles for long runs of waves: with the static
  // round robin, units that run slightly faster drift ahead (at 16384^3 the
  // start of a unit's 40th tile spreads over 120 us, more than a tile), the
  // tiles in flight spread over several waves and their shared operands are
  // evicted from L2 between uses: DRAM reads 18.7 GB per launch static, 11.8
  // GB dynamic, which under the power cap buys SM clock (16384^3 +3 to +5%).
  // Its hand-off costs ~0.5% when the clock is not capped (8192^3: 1908 vs
  // 1898 TFLOP/s, 13 waves), so it is used from 24 waves of whole tiles on.
  // (Mode 2, for testing, uses the machinery whenever there are whole tiles.)
  s.dyn = p->tile_ctr != nullptr && p->tile_order != 1 && vi.ksplit == 1 &&
          (p->tile_order == 2 ? s.dp_tiles > 0 : s.dp_tiles >= 24 * s.units);
  s.grid = static_cast<int>(s.units * vi.ctas);
  return s;
}

template <class Cfg>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                        const GemmArgs& args, int grid, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (Cfg::kClusterCtas > 1) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attr[cfg.numAttrs].val.clusterDim.x = Cfg::kClusterCtas;
    attr[cfg.numAttrs].val.clusterDim.y = 1;
    attr[cfg.numAttrs].val.clusterDim.z = 1;
    ++cfg.numAttrs;
  }
  if (pdl) {
    // The kernel's set-up may overlap the end of the previous kernel in the
    // stream; it waits for that kernel (griddepcontrol.wait) before touching
    // global memory.
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
  }
  return cudaLaunchKernelEx(&cfg, gb300::gemm_tc_kernel<Cfg>, a, b, c, args);
}

// Clusters of the kernel (CTA pairs, or two-pair clusters) resident at once.
template <class Cfg>
int max_active_clusters() {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(Cfg::kClusterCtas, 1, 1);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = Cfg::kClusterCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gb300::gemm_tc_kernel<Cfg>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// C = A x B^T on device buffers.  C's rows are `ldc` elements apart (0: N),
// so a block of a larger C can be written in place (K > 0 only).
gemm_status_t run_device(gemm_plan_s* p, const void* A, const void* B, void* C, int64_t M,
                         int64_t N, int64_t K, gemm_acc_t acc, cudaStream_t stream,
                         int la = GEMM_K_CONTIGUOUS, int lb = GEMM_K_CONTIGUOUS, int64_t ldc = 0) {
  if (ldc == 0) ldc = N;
  if (K == 0) {
    if (ldc != N || !on_device(C, p->device)) return GEMM_ERR_INVALID_ARG;
    const int64_t n16 = M * N * 2 / 16;
    const int64_t blocks = (n16 + 255) / 256;
    gb300::gemm_zero_fill<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0,
                            stream>>>(static_cast<uint4*>(C), n16);
    ++p->launches;
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
  }
  const bool a_mn = la == GEMM_MN_CONTIGUOUS, b_mn = lb == GEMM_MN_CONTIGUOUS;
  // The kernel indexes tiles with 32-bit integers; the smallest tile is
  // 16 x 64, so this bound is far beyond any C that fits in memory.
  if ((M + 15) / 16 * ((N + 63) / 64) > INT32_MAX) return GEMM_ERR_INVALID_ARG;
  const Schedule sch = make_schedule(p, M, N, K, acc, a_mn || b_mn);
  const int grid = sch.grid;
  const VariantInfo& vi = kVariants[sch.variant];
  if (vi.swap && (a_mn || b_mn)) return GEMM_ERR_INVALID_ARG;  // forced swapped variant
  // K-contiguous operands: boxes of 64 K-elements x the tile's rows.
  // M/N-contiguous operands (stored [K, M] / [K, N]): boxes of 64 x 64.
  CUtensorMap ma, mb, mc;
  MapResult mr =
      a_mn ? get_map(p, &ma, A, K, M, 64, 64) : get_map(p, &ma, A, M, K, vi.box_a_rows, 64);
  if (mr == kMapOk)
    mr = b_mn ? get_map(p, &mb, B, K, N, 64, 64) : get_map(p, &mb, B, N, K, vi.box_b_rows, 64);
  if (mr == kMapOk) mr = get_map(p, &mc, C, M, N, 32, 64, static_cast<uint64_t>(ldc));
  if (mr != kMapOk) return mr == kMapNotDevice ? GEMM_ERR_INVALID_ARG : GEMM_ERR_CUDA;

  GemmArgs args;
  args.M = static_cast<int32_t>(M);
  args.N = static_cast<int32_t>(N);
  args.K = static_cast<int32_t>(K);
  if (vi.swap) {
    // The kernel's "A" walks 128-row tiles of B, its "B" tiles of A's rows.
    std::swap(ma, mb);
    args.tiles_m = static_cast<int32_t>((N + vi.tile_n - 1) / vi.tile_n);
    args.tiles_n = static_cast<int32_t>((M + vi.tile_m - 1) / vi.tile_m);
  } else {
    args.tiles_m = static_cast<int32_t>((M + vi.tile_m - 1) / vi.tile_m);
    args.tiles_n = static_cast<int32_t>((N + vi.tile_n - 1) / vi.tile_n);
  }
  args.C = static_cast<uint16_t*>(C);
  args.ldc = ldc;
  args.a_mn = a_mn ? 1 : 0;
  args.b_mn = b_mn ? 1 : 0;
  args.num_kb = static_cast<int32_t>((K + 63) / 64);
  args.num_tiles = args.tiles_m * args.tiles_n;
  args.group_m = kGroupM;
  args.err = p->d_err;
  args.timeout_ns = p->timeout_ns;
  args.skip_kb = p->skip_kb;
  args.dp_tiles = static_cast<int32_t>(sch.dp_tiles);
  args.sk_units = static_cast<int32_t>(sch.sk_units);
  args.sk_iters = sch.sk_iters;
  args.sk_ws = p->sk_ws;
  args.sk_count = p->sk_count;
  args.tile_ctr = sch.dyn ? p->tile_ctr : nullptr;
  args.clk = p->clock_record ? p->d_clk : nullptr;

  const bool f32 = acc == GEMM_ACC_F32;
  cudaError_t e;
  switch (sch.variant) {
    case kVariantPair:
      e = f32 ? launch_gemm<PairF32>(ma, mb, mc, args, grid, stream, p->pdl)
              : launch_gemm<PairF16>(ma, mb, mc, args, grid, stream, p->pdl);
      break;
    case kVariantPairMc:
      e = f32 ? launch_gemm<PairMcF32>(ma, mb, mc, args, grid, stream, p->pdl)
              : launch_gemm<PairMcF16>(ma, mb, mc, args, grid, stream, p->pdl);
      break;
    case kVariantPair128:
      e = f32 ? launch_gemm<Pair128F32>(ma, mb, mc, args, grid, stream, p->pdl)
              : launch_gemm<Pair128F16>(ma, mb, mc, args, grid, stream, p->pdl);
      break;
    case kVariantSingle64:
      e = f32 ? launch_gemm<Single64F32>(ma, mb, mc, args, grid, stream, p->pdl)
              : launch_gemm<Single64F16>(ma, mb, mc, args, grid, stream, p->pdl);
      break;
    case kVariantSwap16:
      e = f32 ? launch_gemm<Swap16F32>(ma, mb, mc, args, grid, stream, p->pdl)
              : launch_gemm<Swap16F16>(ma, mb, mc, args, grid, stream, p->pdl);
      break;
    case kVariantSwap32:
      e = f32 ? launch_gemm<Swap32F32>(ma, mb, mc, args, grid, stream, p->pdl)
              : launch_gemm<Swap32F16>(ma, mb, mc, args, grid, stream, p->pdl);
      break;
    case kVariantSwap64:
      e = f32 ? launch_gemm<Swap64F32>(ma, mb, mc, args, grid, stream, p->pdl)
              : launch_gemm<Swap64F16>(ma, mb, mc, args, grid, stream, p->pdl);
      break;
    // Split-K clusters: fp32 only (make_schedule never picks them for fp16).
    case kVariantSwap16K2:
      e = launch_gemm<Swap16K2F32>(ma, mb, mc, args, grid, stream, p->pdl);
      break;
    case kVariantSwap32K2:
      e = launch_gemm<Swap32K2F32>(ma, mb, mc, args, grid, stream, p->pdl);
      break;
    case kVariantSwap64K2:
      e = launch_gemm<Swap64K2F32>(ma, mb, mc, args, grid, stream, p->pdl);
      break;
    case kVariantSingle64K4:
      e = launch_gemm<Single64K4F32>(ma, mb, mc, args, grid, stream, p->pdl);
      break;
    default:
      e = f32 ? launch_gemm<SingleF32>(ma, mb, mc, args, grid, stream, p->pdl)
              : launch_gemm<SingleF16>(ma, mb, mc, args, grid, stream, p->pdl);
  }
  ++p->launches;
  return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

template <class Cfg>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(gb300::gemm_tc_kernel<Cfg>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
}

gemm_status_t grow(void** buf, size_t* cap, size_t need) {
  if (need <= *cap) return GEMM_OK;
  if (*buf) cudaFree(*buf);
  *buf = nullptr;
  *cap = 0;
  if (cudaMalloc(buf, need) != cudaSuccess) {
    *buf = nullptr;
    return GEMM_ERR_OOM;
  }
  *cap = need;
  return GEMM_OK;
}

}  // namespace

extern "C" {

const char* gemm_version(void) { return GB300_GEMM_VERSION; }

const char* gemm_status_string(gemm_status_t s) {
  switch (s) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
    case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT";
    case GEMM_ERR_UNSUPPORTED_DEVICE: return "GEMM_ERR_UNSUPPORTED_DEVICE";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    case GEMM_ERR_OOM: return "GEMM_ERR_OOM";
  }
  return "GEMM_ERR_UNKNOWN";
}

int32_t gemm_variant_count(void) { return kNumVariants; }

int32_t gemm_variant_info(int32_t v, int32_t out[4]) {
  if (v < 0 || v >= kNumVariants || !out) return -1;
  out[0] = kVariants[v].ctas;
  out[1] = kVariants[v].tile_m;
  out[2] = kVariants[v].tile_n;
  out[3] = kVariants[v].swap ? 1 : 0;
  return 0;
}

gemm_status_t gemm_plan_resident_units(gemm_plan_t p, int32_t out[3]) {
  if (!p || !out) return GEMM_ERR_INVALID_ARG;
  out[0] = p->num_sms;
  out[1] = p->max_pairs;
  out[2] = p->max_quads;
  return GEMM_OK;
}

const char* gemm_variant_name(int32_t v) {
  return (v >= 0 && v < kNumVariants) ? kVariants[v].name : nullptr;
}

gemm_status_t gemm_plan_create(gemm_plan_t* out, int device) {
  if (!out) return GEMM_ERR_INVALID_ARG;
  *out = nullptr;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) return GEMM_ERR_CUDA;
  if (device < 0 || device >= ndev) return GEMM_ERR_INVALID_ARG;
  DeviceGuard g(device);
  if (!g.ok) return GEMM_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return GEMM_ERR_CUDA;
  if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED_DEVICE;

  gemm_plan_s* p = new (std::nothrow) gemm_plan_s();
  if (!p) return GEMM_ERR_OOM;
  std::memset(p->maps, 0, sizeof(p->maps));
  p->device = device;
  p->num_sms = sms;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    delete p;
    return GEMM_ERR_CUDA;
  }
  p->encode = reinterpret_cast<EncodeTiledFn>(fn);
  if (set_smem_attr<SingleF32>() != cudaSuccess || set_smem_attr<SingleF16>() != cudaSuccess ||
      set_smem_attr<PairF32>() != cudaSuccess || set_smem_attr<PairF16>() != cudaSuccess ||
      set_smem_attr<Pair128F32>() != cudaSuccess || set_smem_attr<Pair128F16>() != cudaSuccess ||
      set_smem_attr<Single64F32>() != cudaSuccess || set_smem_attr<Single64F16>() != cudaSuccess ||
      set_smem_attr<Swap16F32>() != cudaSuccess || set_smem_attr<Swap16F16>() != cudaSuccess ||
      set_smem_attr<Swap32F32>() != cudaSuccess || set_smem_attr<Swap32F16>() != cudaSuccess ||
      set_smem_attr<Swap64F32>() != cudaSuccess || set_smem_attr<Swap64F16>() != cudaSuccess ||
      set_smem_attr<PairMcF32>() != cudaSuccess || set_smem_attr<PairMcF16>() != cudaSuccess ||
      set_smem_attr<Swap16K2F32>() != cudaSuccess || set_smem_attr<Swap32K2F32>() != cudaSuccess ||
      set_smem_attr<Swap64K2F32>() != cudaSuccess || set_smem_attr<Single64K4F32>() != cudaSuccess) {
    delete p;
    return GEMM_ERR_CUDA;
  }
  {
    int m = max_active_clusters<PairF32>();
    for (int n : {max_active_clusters<PairF16>(), max_active_clusters<Pair128F32>(),
                  max_active_clusters<Pair128F16>()})
      m = n < m ? n : m;
    p->max_pairs = m;
    const int q0 = max_active_clusters<PairMcF32>(), q1 = max_active_clusters<PairMcF16>();
    p->max_quads = q0 < q1 ? q0 : q1;
    for (int v = 0; v < kNumVariants; ++v) {
      const int c = kVariants[v].ctas;
      p->max_units[v] = c == 4 ? p->max_quads : c == 2 ? p->max_pairs : p->num_sms;
    }
    p->max_units[kVariantSwap16K2] = max_active_clusters<Swap16K2F32>();
    p->max_units[kVariantSwap32K2] = max_active_clusters<Swap32K2F32>();
    p->max_units[kVariantSwap64K2] = max_active_clusters<Swap64K2F32>();
    p->max_units[kVariantSingle64K4] = max_active_clusters<Single64K4F32>();
  }
  // 16-byte watchdog record, then three 8-byte clock counters.
  if (cudaMalloc(&p->d_err, kRecordBytes) != cudaSuccess) {
    delete p;
    return GEMM_ERR_OOM;
  }
  p->d_clk = reinterpret_cast<unsigned long long*>(p->d_err + 4);
  if (cudaMemset(p->d_err, 0, kRecordBytes) != cudaSuccess) {
    cudaFree(p->d_err);
    delete p;
    return GEMM_ERR_CUDA;
  }
  // Stream-K workspace: two 128 x 256 fp32 partial tiles per CTA the device
  // can hold at once (≈ 39 MB on 152 SMs), and up to two tail tiles per unit.
  {
    const size_t ws_floats = 2ull * static_cast<size_t>(sms) * 128ull * 256ull;
    p->sk_count_words = 4ull * static_cast<size_t>(sms);
    if (cudaMalloc(&p->sk_ws, ws_floats * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&p->sk_count, (p->sk_count_words + 2) * sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(p->sk_count, 0, (p->sk_count_words + 2) * sizeof(uint32_t)) != cudaSuccess) {
      if (p->sk_ws) cudaFree(p->sk_ws);
      if (p->sk_count) cudaFree(p->sk_count);
      cudaFree(p->d_err);
      delete p;
      return GEMM_ERR_OOM;
    }
    p->tile_ctr = p->sk_count + p->sk_count_words;
  }
  *out = p;
  return GEMM_OK;
}

gemm_status_t gemm_plan_destroy(gemm_plan_t p) {
  if (!p) return GEMM_OK;
  DeviceGuard g(p->device);
  if (p->d_err) cudaFree(p->d_err);
  if (p->sk_ws) cudaFree(p->sk_ws);
  if (p->sk_count) cudaFree(p->sk_count);
  for (cudaStream_t st : {p->s_in, p->s_comp, p->s_out})
    if (st) cudaStreamDestroy(st);
  if (p->ev_start) cudaEventDestroy(p->ev_start);
  for (cudaEvent_t e : p->ev_in)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : p->ev_comp)
    if (e) cudaEventDestroy(e);
  if (p->dA) cudaFree(p->dA);
  if (p->dB) cudaFree(p->dB);
  if (p->dC) cudaFree(p->dC);
  delete p;
  return GEMM_OK;
}

gemm_status_t gemm_plan_set_watchdog(gemm_plan_t p, uint64_t timeout_ns, int32_t skip_k_block) {
  if (!p || skip_k_block < -1) return GEMM_ERR_INVALID_ARG;
  p->timeout_ns = timeout_ns ? timeout_ns : kDefaultTimeoutNs;
  p->skip_kb = skip_k_block;
  return GEMM_OK;
}

gemm_status_t gemm_plan_set_schedule(gemm_plan_t p, int32_t mode) {
  if (!p || mode < 0 || mode > 2) return GEMM_ERR_INVALID_ARG;
  p->schedule_mode = mode;
  return GEMM_OK;
}

int32_t gemm_plan_describe(gemm_plan_t p, int64_t M, int64_t N, int64_t K, gemm_acc_t acc,
                           int64_t out[6]) {
  if (!p || !out || check_shape(M, N, K, acc) != GEMM_OK) return -1;
  const Schedule s = make_schedule(p, M, N, K, acc);
  out[0] = s.variant;
  out[1] = s.grid;
  out[2] = s.units;
  out[3] = s.dp_tiles;
  out[4] = s.sk_units;
  out[5] = s.sk_iters;
  return 0;
}

gemm_status_t gemm_plan_set_tile_order(gemm_plan_t p, int32_t mode) {
  if (!p || mode < 0 || mode > 2) return GEMM_ERR_INVALID_ARG;
  p->tile_order = mode;
  return GEMM_OK;
}

gemm_status_t gemm_plan_set_clock_record(gemm_plan_t p, int32_t enable) {
  if (!p || (enable != 0 && enable != 1)) return GEMM_ERR_INVALID_ARG;
  p->clock_record = enable != 0;
  return GEMM_OK;
}

gemm_status_t gemm_plan_set_pdl(gemm_plan_t p, int32_t enable) {
  if (!p || (enable != 0 && enable != 1)) return GEMM_ERR_INVALID_ARG;
  p->pdl = enable != 0;
  return GEMM_OK;
}

gemm_status_t gemm_plan_set_variant(gemm_plan_t p, int32_t v) {
  if (!p || v < -1 || v >= kNumVariants) return GEMM_ERR_INVALID_ARG;
  p->forced_variant = v;
  return GEMM_OK;
}

int32_t gemm_plan_pick_variant(gemm_plan_t p, int64_t M, int64_t N, int64_t K, gemm_acc_t acc,
                               int32_t* grid_ctas) {
  if (!p || check_shape(M, N, K, acc) != GEMM_OK) return -1;
  const Schedule s = make_schedule(p, M, N, K, acc);
  if (grid_ctas) *grid_ctas = s.grid;
  return s.variant;
}

uint64_t gemm_plan_launch_count(gemm_plan_t p) { return p ? p->launches : 0; }

gemm_status_t gemm_run(gemm_plan_t p, const void* A, const void* B, void* C, int64_t M, int64_t N,
                       int64_t K, gemm_acc_t acc, void* stream) {
  if (!p) return GEMM_ERR_INVALID_ARG;
  gemm_status_t s = check_shape(M, N, K, acc);
  if (s != GEMM_OK) return s;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(C) & 15) ||
      (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15))))
    return GEMM_ERR_ALIGNMENT;
  const size_t bytesC = static_cast<size_t>(M) * N * 2;
  if (K > 0 && (overlaps(C, bytesC, A, static_cast<size_t>(M) * K * 2) ||
                overlaps(C, bytesC, B, static_cast<size_t>(N) * K * 2)))
    return GEMM_ERR_INVALID_ARG;
  DeviceGuard g(p->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  return run_device(p, A, B, C, M, N, K, acc, static_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_run_ex(gemm_plan_t p, const void* A, gemm_layout_t layout_a, const void* B,
                          gemm_layout_t layout_b, void* C, int64_t M, int64_t N, int64_t K,
                          gemm_acc_t acc, void* stream) {
  if (!p) return GEMM_ERR_INVALID_ARG;
  const bool la_ok = layout_a == GEMM_K_CONTIGUOUS || layout_a == GEMM_MN_CONTIGUOUS;
  const bool lb_ok = layout_b == GEMM_K_CONTIGUOUS || layout_b == GEMM_MN_CONTIGUOUS;
  if (!la_ok || !lb_ok) return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
    return GEMM_ERR_INVALID_ARG;
  if (acc != GEMM_ACC_F32 && acc != GEMM_ACC_F16) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  // Every stored row must start on a 16-byte boundary: the contiguous
  // dimension of each operand, and N for C, is a multiple of 8.
  if (N % 8 != 0) return GEMM_ERR_ALIGNMENT;
  if ((layout_a == GEMM_K_CONTIGUOUS || layout_b == GEMM_K_CONTIGUOUS) && K % 8 != 0)
    return GEMM_ERR_ALIGNMENT;
  if (layout_a == GEMM_MN_CONTIGUOUS && M % 8 != 0) return GEMM_ERR_ALIGNMENT;
  if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(C) & 15) ||
      (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15))))
    return GEMM_ERR_ALIGNMENT;
  const size_t bytesC = static_cast<size_t>(M) * N * 2;
  if (K > 0 && (overlaps(C, bytesC, A, static_cast<size_t>(M) * K * 2) ||
                overlaps(C, bytesC, B, static_cast<size_t>(N) * K * 2)))
    return GEMM_ERR_INVALID_ARG;
  DeviceGuard g(p->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  return run_device(p, A, B, C, M, N, K, acc, static_cast<cudaStream_t>(stream), layout_a,
                    layout_b);
}

gemm_status_t gemm_plan_check_error(gemm_plan_t p) {
  if (!p) return GEMM_ERR_INVALID_ARG;
  DeviceGuard g(p->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  uint32_t rec[4] = {0, 0, 0, 0};
  if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
  if (cudaMemcpy(rec, p->d_err, sizeof(rec), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GEMM_ERR_CUDA;
  if (rec[0] == 0) return GEMM_OK;
  std::memcpy(p->last_err, rec, sizeof(rec));
  if (cudaMemset(p->d_err, 0, sizeof(rec)) != cudaSuccess) return GEMM_ERR_CUDA;
  // A launch that gave up may have left the stream-K and tile-order
  // counters mid-count.
  if (p->sk_count &&
      cudaMemset(p->sk_count, 0, (p->sk_count_words + 2) * sizeof(uint32_t)) != cudaSuccess)
    return GEMM_ERR_CUDA;
  return static_cast<gemm_status_t>(rec[0]);
}

gemm_status_t gemm_plan_last_error_detail(gemm_plan_t p, uint32_t detail[4]) {
  if (!p || !detail) return GEMM_ERR_INVALID_ARG;
  std::memcpy(detail, p->last_err, sizeof(p->last_err));
  return GEMM_OK;
}

gemm_status_t gemm_plan_kernel_clock(gemm_plan_t p, uint64_t out[3]) {
  if (!p || !out) return GEMM_ERR_INVALID_ARG;
  DeviceGuard g(p->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  unsigned long long rec[3] = {0, 0, 0};
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(rec, p->d_clk, sizeof(rec), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(p->d_clk, 0, sizeof(rec)) != cudaSuccess)
    return GEMM_ERR_CUDA;
  for (int i = 0; i < 3; ++i) out[i] = static_cast<uint64_t>(rec[i]);
  return GEMM_OK;
}

gemm_status_t gemm_run_host(gemm_plan_t p, const void* A, const void* B, void* C, int64_t M,
                            int64_t N, int64_t K, gemm_acc_t acc, void* stream) {
  if (!p) return GEMM_ERR_INVALID_ARG;
  gemm_status_t s = check_shape(M, N, K, acc);
  if (s != GEMM_OK) return s;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
  DeviceGuard g(p->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  const size_t bA = static_cast<size_t>(M) * K * 2, bB = static_cast<size_t>(N) * K * 2,
               bC = static_cast<size_t>(M) * N * 2;
  if ((s = grow(&p->dA, &p->capA, bA > 0 ? bA : 16)) != GEMM_OK) return s;
  if ((s = grow(&p->dB, &p->capB, bB > 0 ? bB : 16)) != GEMM_OK) return s;
  if ((s = grow(&p->dC, &p->capC, bC)) != GEMM_OK) return s;
  if (!p->s_in) {
    bool ok = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->s_comp, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->ev_start, cudaEventDisableTiming) == cudaSuccess;
    for (cudaEvent_t& e : p->ev_in)
      ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
    for (cudaEvent_t& e : p->ev_comp)
      ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return GEMM_ERR_CUDA;
  }
  auto& d = *p;
  bool ok = cudaEventRecord(d.ev_start, static_cast<cudaStream_t>(stream)) == cudaSuccess &&
            cudaStreamWaitEvent(d.s_in, d.ev_start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(d.s_comp, d.ev_start, 0) == cudaSuccess;
  if (ok && K == 0) {  // the empty sum: zeros, no input to copy
    ok = (s = run_device(p, nullptr, nullptr, d.dC, M, N, 0, acc, d.s_comp)) == GEMM_OK &&
         cudaEventRecord(d.ev_comp[0], d.s_comp) == cudaSuccess &&
         cudaStreamWaitEvent(d.s_out, d.ev_comp[0], 0) == cudaSuccess &&
         cudaMemcpyAsync(C, d.dC, bC, cudaMemcpyDeviceToHost, d.s_out) == cudaSuccess;
  }
  // The pipeline.  A is cut into row chunks A_i and B into row chunks B_j
  // (whole 256-row tiles); the copy-in stream sends them alternately, in
  // proportion, block C_ij = A_i B_j^T is multiplied as soon as both of its
  // chunks have arrived, and the copy-out stream returns each block (a
  // strided 2-D copy) while later chunks are still coming in, so both
  // directions of the host link and the tensor cores overlap.  Work starts
  // after everything already queued on the caller's stream.
  // Compute time over copy-in time goes as MN / (M + N), whatever K.  Below
  // ~6144 the host link is the bound: B whole and A in chunks of at most
  // 1024 rows (at least four), so only the first and last chunk are exposed
  // (8192^3: 662 TFLOP/s; cutting B too gave 664, 4096^3 277 vs 294).  Above
  // it the tensor cores matter as much, and cutting both operands into
  // ~2048-row chunks lets them start after two chunks instead of all of B
  // (16384^3: 1252 vs 1086).
  auto tiles256 = [](int64_t r) { return (r + 255) / 256 * 256; };
  int64_t rows = 0, cols = 0;
  int mc = 0, nc = 0;
  if (K > 0) {
    if (static_cast<double>(M) * static_cast<double>(N) / static_cast<double>(M + N) >= 6144.0) {
      auto split = [&](int64_t n, int64_t& per) {
        const int64_t parts = std::min<int64_t>(kHostChunksB, std::max<int64_t>(1, (n + 1024) / 2048));
        per = tiles256((n + parts - 1) / parts);
        return static_cast<int>((n + per - 1) / per);
      };
      mc = split(M, rows);
      nc = split(N, cols);
    } else {
      rows = std::min<int64_t>(1024, tiles256((M + 3) / 4));
      rows = std::max<int64_t>(rows, tiles256((M + kHostChunksA - 1) / kHostChunksA));
      mc = static_cast<int>((M + rows - 1) / rows);
      cols = N;
      nc = 1;
    }
  }
  bool have_a[kHostChunksA] = {}, have_b[kHostChunksB] = {};
  int ia = 0, ib = 0, blocks = 0;
  for (int step = 0; ok && step < mc + nc; ++step) {
    // Next chunk: the operand with the smaller fraction sent so far.
    const bool take_a = ib == nc || (ia < mc && static_cast<int64_t>(ia) * nc <= static_cast<int64_t>(ib) * mc);
    const int idx = take_a ? ia++ : ib++;
    const int64_t r0 = idx * (take_a ? rows : cols);
    const int64_t n = std::min<int64_t>(take_a ? rows : cols, (take_a ? M : N) - r0);
    const char* src = static_cast<const char*>(take_a ? A : B) + r0 * K * 2;
    char* dst = static_cast<char*>(take_a ? d.dA : d.dB) + r0 * K * 2;
    ok = cudaMemcpyAsync(dst, src, static_cast<size_t>(n) * K * 2, cudaMemcpyHostToDevice, d.s_in) ==
             cudaSuccess &&
         cudaEventRecord(d.ev_in[step], d.s_in) == cudaSuccess &&
         cudaStreamWaitEvent(d.s_comp, d.ev_in[step], 0) == cudaSuccess;
    (take_a ? have_a : have_b)[idx] = true;
    // Every block this chunk completes.
    for (int other = 0; ok && other < (take_a ? nc : mc); ++other) {
      if (!(take_a ? have_b : have_a)[other]) continue;
      const int i = take_a ? idx : other, j = take_a ? other : idx;
      const int64_t m0 = i * rows, mi = std::min<int64_t>(rows, M - m0);
      const int64_t n0 = j * cols, nj = std::min<int64_t>(cols, N - n0);
      const size_t c_off = static_cast<size_t>(m0 * N + n0) * 2;
      if ((s = run_device(p, static_cast<char*>(d.dA) + m0 * K * 2,
                          static_cast<char*>(d.dB) + n0 * K * 2, static_cast<char*>(d.dC) + c_off, mi,
                          nj, K, acc, d.s_comp, GEMM_K_CONTIGUOUS, GEMM_K_CONTIGUOUS, N)) != GEMM_OK) {
        ok = false;
        break;
      }
      cudaEvent_t e = d.ev_comp[blocks++];
      ok = cudaEventRecord(e, d.s_comp) == cudaSuccess &&
           cudaStreamWaitEvent(d.s_out, e, 0) == cudaSuccess &&
           cudaMemcpy2DAsync(static_cast<char*>(C) + c_off, N * 2, static_cast<char*>(d.dC) + c_off,
                             N * 2, nj * 2, mi, cudaMemcpyDeviceToHost, d.s_out) == cudaSuccess;
    }
  }
  const bool synced = cudaStreamSynchronize(d.s_in) == cudaSuccess &&
                      cudaStreamSynchronize(d.s_comp) == cudaSuccess &&
                      cudaStreamSynchronize(d.s_out) == cudaSuccess;
  if (s != GEMM_OK) return s;
  if (!ok || !synced) return GEMM_ERR_CUDA;
  uint32_t code = 0;
  if (cudaMemcpy(&code, p->d_err, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GEMM_ERR_CUDA;
  return code == 0 ? GEMM_OK : gemm_plan_check_error(p);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot call cudaMalloc: code running under an allocator that
// owns every byte of device memory (a framework's caching allocator, or a
// fixed arena carved out at start-up, where a stray cudaMalloc can fail or
// fragment the pool), and latency-bound loops where cudaMalloc's implicit
// device synchronisation would stall other streams.  gemm_plan_create
// allocates the kernel's watchdog record with cudaMalloc, so such callers
// cannot make a plan.  gemm_run_noalloc runs the same kernel with that
// scratch -- the 16-byte watchdog record, the only global memory the kernel
// touches beyond A, B and C -- in the file-scope array below instead.
//
// The array is a static device variable: every GPU that loads this library
// holds its 256 bytes until the process exits.  In host code its name is only
// a host-side stand-in, never a device address, so each device's address is
// looked up once with cudaGetSymbolAddress (with that device current) and
// that address is what the kernel receives.
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(uint32_t)];

namespace {

constexpr int kNoAllocMaxDevices = 64;
// Scratch the single-CTA kernel needs for one call, whatever the shape.
constexpr size_t kNoAllocRecordBytes = 4 * sizeof(uint32_t);

struct NoAllocDevice {
  std::once_flag once;
  gemm_status_t status = GEMM_ERR_CUDA;
  int num_sms = 0;
  uint32_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::once_flag g_noalloc_encode_once;
EncodeTiledFn g_noalloc_encode = nullptr;

// One-time set-up for the current device `dev`.
gemm_status_t noalloc_setup(int dev, NoAllocDevice& d) {
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GEMM_ERR_CUDA;
  if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED_DEVICE;
  std::call_once(g_noalloc_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_noalloc_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (!g_noalloc_encode) return GEMM_ERR_CUDA;
  if (set_smem_attr<SingleF32>() != cudaSuccess || set_smem_attr<SingleF16>() != cudaSuccess)
    return GEMM_ERR_CUDA;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return GEMM_ERR_CUDA;
  d.scratch = static_cast<uint32_t*>(ptr);
  d.num_sms = sms;
  return GEMM_OK;
}

bool noalloc_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                 uint32_t box_rows, uint32_t box_cols) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_noalloc_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, l2_promotion(cols * 2),
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" gemm_status_t gemm_run_noalloc(const void* A, const void* B, void* C, int64_t M,
                                          int64_t N, int64_t K, gemm_acc_t acc, void* stream) {
  gemm_status_t s = check_shape(M, N, K, acc);
  if (s != GEMM_OK) return s;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(C) & 15) ||
      (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15))))
    return GEMM_ERR_ALIGNMENT;
  const size_t bytesC = static_cast<size_t>(M) * N * 2;
  if (K > 0 && (overlaps(C, bytesC, A, static_cast<size_t>(M) * K * 2) ||
                overlaps(C, bytesC, B, static_cast<size_t>(N) * K * 2)))
    return GEMM_ERR_INVALID_ARG;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return GEMM_ERR_CUDA;
  if (dev >= kNoAllocMaxDevices) return GEMM_ERR_INVALID_ARG;
  if (!on_device(C, dev) || (K > 0 && (!on_device(A, dev) || !on_device(B, dev))))
    return GEMM_ERR_INVALID_ARG;
  NoAllocDevice& d = g_noalloc_dev[dev];
  std::call_once(d.once, [&] { d.status = noalloc_setup(dev, d); });
  if (d.status != GEMM_OK) return d.status;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) {  // the empty sum: zeros, no scratch involved
    const int64_t n16 = M * N * 2 / 16;
    const int64_t blocks = (n16 + 255) / 256;
    gb300::gemm_zero_fill<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(
        static_cast<uint4*>(C), n16);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
  }
  // The scratch this call needs must fit the array.
  if (kNoAllocRecordBytes > kNoAllocScratchBytes) return GEMM_ERR_INVALID_ARG;

  const VariantInfo& vi = kVariants[kVariantSingle];
  CUtensorMap ma, mb, mc;
  if (!noalloc_map(&ma, A, M, K, vi.box_a_rows, 64) || !noalloc_map(&mb, B, N, K, vi.box_b_rows, 64) ||
      !noalloc_map(&mc, C, M, N, 32, 64))
    return GEMM_ERR_CUDA;
  GemmArgs args;
  args.M = static_cast<int32_t>(M);
  args.N = static_cast<int32_t>(N);
  args.K = static_cast<int32_t>(K);
  args.tiles_m = static_cast<int32_t>((M + vi.tile_m - 1) / vi.tile_m);
  args.tiles_n = static_cast<int32_t>((N + vi.tile_n - 1) / vi.tile_n);
  args.num_kb = static_cast<int32_t>((K + 63) / 64);
  args.num_tiles = args.tiles_m * args.tiles_n;
  args.group_m = kGroupM;
  args.err = d.scratch;
  args.timeout_ns = kDefaultTimeoutNs;
  args.skip_kb = -1;
  args.dp_tiles = args.num_tiles;  // whole tiles only: no stream-K workspace here
  args.sk_units = 0;
  args.sk_iters = 0;
  args.sk_ws = nullptr;
  args.sk_count = nullptr;
  args.tile_ctr = nullptr;  // static tile order: no counters here
  args.clk = nullptr;       // no clock record either
  args.C = static_cast<uint16_t*>(C);
  args.ldc = N;
  args.a_mn = 0;
  args.b_mn = 0;
  const int grid = args.num_tiles < d.num_sms ? args.num_tiles : d.num_sms;
  // The watchdog record must start at zero; the array keeps the last call's
  // contents, so clear it on the caller's stream before the launch.
  if (cudaMemsetAsync(d.scratch, 0, kNoAllocRecordBytes, st) != cudaSuccess) return GEMM_ERR_CUDA;
  cudaError_t e = acc == GEMM_ACC_F32 ? launch_gemm<SingleF32>(ma, mb, mc, args, grid, st, false)
                                      : launch_gemm<SingleF16>(ma, mb, mc, args, grid, st, false);
  return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
