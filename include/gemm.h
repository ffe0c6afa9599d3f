/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense fp16 GEMM library.
 *
 * The operation (tilus "A Minimal Hopper Matmul", section "Block Tiling", and
 * its note "Data layout: K-major"):
 *
 *     C[M, N] = A[M, K] x B[N, K]^T,    C[i][j] = sum_k A[i][k] * B[j][k]
 *
 * A, B and C are fp16 (IEEE binary16), row-major, K contiguous in A and B.
 * The sum runs on the tensor cores (tcgen05.mma, accumulator in tensor
 * memory), accumulated in fp32 (GEMM_ACC_F32) or natively in fp16
 * (GEMM_ACC_F16, tilus "Four Consumers, FP16 Accumulation, and a TMA
 * Epilogue", section "The Register Budget Problem"), and written as fp16
 * rounded to nearest even.
 *
 * Ownership: the caller owns every buffer.  The library owns only the plan:
 * the device watchdog record, a stream-K workspace of about 0.25 MB per SM
 * (allocated when the plan is created), and, for gemm_run_host, device staging
 * buffers it grows on demand.
 *
 * Errors: every entry point returns a gemm_status_t.  Argument checks run on
 * the host before any launch, so a rejected call writes nothing.  A kernel
 * that stops making progress (a wait that outlives the plan's timeout) does
 * not hang: it records GEMM_ERR_TIMEOUT on the device, frees its tensor
 * memory and returns; gemm_plan_check_error reports it.
 *
 * Threads and streams: a plan may be used by one host thread at a time, and
 * work launched through one plan must not run concurrently on the GPU (its
 * calls share the plan's workspace): give each stream its own plan.
 * Different plans are independent.
 */
#ifndef GB300_GEMM_H_
#define GB300_GEMM_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemm_plan_s* gemm_plan_t;

/* Accumulation precision inside the tensor cores. */
typedef enum {
    GEMM_ACC_F32 = 0, /* fp32 accumulate, fp16 output (the default) */
    GEMM_ACC_F16 = 1  /* native fp16 accumulate, fp16 output */
} gemm_acc_t;

/* Storage of an operand (gemm_run_ex).  Logically A is M x K and B is N x K
 * whatever the storage:
 *   GEMM_K_CONTIGUOUS : A stored [M, K], B stored [N, K] (rows along K; the
 *                       layout of gemm_run)
 *   GEMM_MN_CONTIGUOUS: A stored [K, M] (A(m,k) at A[k*M + m]), B stored
 *                       [K, N] (B(n,k) at B[k*N + n]); with B so stored the
 *                       call computes the usual row-major C = A x B.
 * The tensor cores read both forms directly (tilus "A Minimal Hopper
 * Matmul", "Block Tiling", note "Data layout: K-major": operands may be
 * K-contiguous or MN-contiguous). */
typedef enum {
    GEMM_K_CONTIGUOUS = 0,
    GEMM_MN_CONTIGUOUS = 1
} gemm_layout_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,        /* null plan/pointer, negative or oversized dim, bad enum, C overlaps A or B */
    GEMM_ERR_ALIGNMENT = 2,          /* pointer not 16-byte aligned, K or N not a multiple of 8 */
    GEMM_ERR_UNSUPPORTED_DEVICE = 3, /* device is not compute capability 10.3 (sm_103a) */
    GEMM_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed (launch, copy, allocation of plan memory) */
    GEMM_ERR_TIMEOUT = 5,            /* the kernel's watchdog fired: a wait outlived the plan's timeout */
    GEMM_ERR_OOM = 6                 /* host or device memory for the plan could not be allocated */
} gemm_status_t;

/* Create a plan bound to CUDA device `device` (must be an sm_103 part).
 * Queries the SM count, resolves the tensor-map encoder from the driver, sets
 * the kernels' shared-memory limits and allocates a 64-byte device record
 * (the kernel's watchdog and clock records) and the stream-K workspace.  *out receives the plan, or NULL on error. */
GEMM_API gemm_status_t gemm_plan_create(gemm_plan_t* out, int device);

/* Release the plan and everything it allocated.  NULL is accepted (no-op).
 * Must not be called while work launched with the plan is still running. */
GEMM_API gemm_status_t gemm_plan_destroy(gemm_plan_t plan);

/* C = A x B^T on device buffers, asynchronously on `stream` (a cudaStream_t
 * of the plan's device; NULL = legacy default stream).  A, B and C must be
 * device memory of the plan's device (cudaMalloc, cudaMallocAsync or virtual
 * memory mapped there): a pointer is looked up with cudaPointerGetAttributes
 * the first time the plan sees it with a given shape (the plan caches the
 * tensor map it then builds), and host, managed or unregistered memory, or
 * another GPU's memory, is refused with GEMM_ERR_INVALID_ARG before any
 * launch.  (Memory freed and allocated again at the same address is not
 * looked up again while its map stays in the plan's cache of 1024 maps.)
 *   A : device pointer, fp16 [M, K] row-major (K contiguous), 16-byte aligned
 *   B : device pointer, fp16 [N, K] row-major (K contiguous), 16-byte aligned
 *   C : device pointer, fp16 [M, N] row-major, 16-byte aligned, must not
 *       overlap A or B
 *   M, N, K : 0 <= M, N, K <= 2^31 - 1;  K % 8 == 0 and N % 8 == 0 (every
 *       row starts on a 16-byte boundary, as the tensor-memory-access engine
 *       requires).  M == 0 or N == 0: nothing to do, GEMM_OK, pointers
 *       unused.  K == 0: C is filled with +0 (the empty sum).
 *   acc : GEMM_ACC_F32 or GEMM_ACC_F16.
 * Allocates nothing, does not synchronize.  Launch failures return
 * GEMM_ERR_CUDA; a device-side watchdog timeout surfaces later through
 * gemm_plan_check_error. */
GEMM_API gemm_status_t gemm_run(gemm_plan_t plan, const void* A, const void* B, void* C,
                       int64_t M, int64_t N, int64_t K, gemm_acc_t acc,
                       void* stream);

/* gemm_run with a choice of storage for each operand (see gemm_layout_t).
 * Alignment rules: N % 8 == 0 always (rows of C); K % 8 == 0 if either
 * operand is K-contiguous; M % 8 == 0 if A is M-contiguous; pointers 16-byte
 * aligned.  Otherwise as gemm_run (device memory of the plan's device,
 * asynchronous, allocates nothing). */
GEMM_API gemm_status_t gemm_run_ex(gemm_plan_t plan, const void* A, gemm_layout_t layout_a,
                                   const void* B, gemm_layout_t layout_b, void* C,
                                   int64_t M, int64_t N, int64_t K, gemm_acc_t acc,
                                   void* stream);

/* Same product on HOST buffers, synchronous: copies row chunks of A and B
 * to device staging buffers owned by the plan (grown with cudaMalloc on
 * first use of a larger shape), multiplies each block of C as soon as the
 * chunks it needs have arrived, and copies the block back while later
 * chunks are still in flight (three internal streams, created on first
 * use).  B travels whole unless M*N/(M+N) >= 6144, when the multiplies are
 * long enough to start them before all of B has arrived.  The work starts
 * after everything already queued on `stream`; the call returns when C is
 * filled.  A, B, C are host pointers (pinned memory gives full copy
 * bandwidth and the overlap; pageable memory works but is slower).  Same
 * shape and alignment rules as gemm_run (host pointers need no particular
 * alignment).  Returns the watchdog status of the run as well. */
GEMM_API gemm_status_t gemm_run_host(gemm_plan_t plan, const void* A, const void* B, void* C,
                            int64_t M, int64_t N, int64_t K, gemm_acc_t acc,
                            void* stream);

/* Synchronize the plan's device, read and clear the watchdog record.
 * Returns GEMM_OK, GEMM_ERR_TIMEOUT (the record is then described by
 * gemm_plan_last_error_detail) or GEMM_ERR_CUDA if the context is broken. */
GEMM_API gemm_status_t gemm_plan_check_error(gemm_plan_t plan);

/* The last watchdog record read by gemm_plan_check_error:
 * detail[0] = status code, detail[1] = which wait gave up (see the kernel's
 * WaitSite list), detail[2] = CTA index, detail[3] = tile index. */
GEMM_API gemm_status_t gemm_plan_last_error_detail(gemm_plan_t plan, uint32_t detail[4]);

/* The SM clock the kernels actually ran at.  While the plan's clock record
 * is on (gemm_plan_set_clock_record), every GEMM kernel launched through the
 * plan has its first CTA add 1, its lifetime in SM cycles (%clock64) and its
 * lifetime in nanoseconds (%globaltimer) to a device record; this call
 * synchronizes the device, copies the record to out[0] = launches,
 * out[1] = cycles, out[2] = ns, and sets it back to zero.  out[1] * 1000 / out[2] is the mean SM clock in MHz over those
 * launches (a clock sampled from outside, e.g. by NVML, can miss the drop a
 * power-capped kernel causes).  gemm_run_host's launches count too; the
 * K == 0 zero-fill does not.  No counterpart in the source pages (a
 * measurement aid). */
GEMM_API gemm_status_t gemm_plan_kernel_clock(gemm_plan_t plan, uint64_t out[3]);

/* Clock record on (1) or off (0, the default).  The record's three atomics
 * at the end of the first CTA lengthen a launch of a few microseconds by
 * ~0.15 us (512^3 in a CUDA graph: 4.30 vs 4.15 us per GEMM); measurement
 * turns it on.  GEMM_ERR_INVALID_ARG for other values.  No counterpart in
 * the source pages (a measurement aid). */
GEMM_API gemm_status_t gemm_plan_set_clock_record(gemm_plan_t plan, int32_t enable);

/* Watchdog and fault-injection controls (testing and diagnosis).
 * timeout_ns: how long any one wait inside the kernel may take before it
 *   gives up (default 2e9 ns; 0 restores the default).
 * skip_k_block: -1 (default) for normal operation; a value >= 0 makes the
 *   producer skip the load of that k-block of the first tile of CTA 0 and
 *   never declare its bytes, so the consumer's wait for it can only end by
 *   timing out.  Used to test that a stuck wait returns an error and leaves
 *   the context usable. */
GEMM_API gemm_status_t gemm_plan_set_watchdog(gemm_plan_t plan, uint64_t timeout_ns,
                                     int32_t skip_k_block);

/* Work schedule: 0 = automatic (default); 1 = whole tiles only; 2 = use the
 * stream-K tail whenever the shape allows it, down to one k-block per CTA
 * (testing).  With the tail, the
 * k-blocks of the last tiles are shared out evenly over all CTAs and partial
 * fp32 tiles are summed in a fixed order in the plan's workspace (so results
 * stay deterministic); fp16 accumulation always uses whole tiles. */
GEMM_API gemm_status_t gemm_plan_set_schedule(gemm_plan_t plan, int32_t mode);

/* Order of whole tiles (a work-scheduling detail; results never depend on
 * it): 0 = automatic (default: dynamic from 24 waves of whole tiles on,
 * e.g. 16384^3), 1 = static round robin over the persistent units, 2 =
 * dynamic whenever there are whole tiles (testing).  In the dynamic order
 * each unit's first whole tile is fixed and the rest are taken from a
 * global ticket counter in the plan as the unit needs them, so tiles start
 * in order across units and the tiles in flight stay within about one wave
 * (their shared operands stay in L2).  GEMM_ERR_INVALID_ARG for other
 * values.  No counterpart in the source pages (a scheduling detail). */
GEMM_API gemm_status_t gemm_plan_set_tile_order(gemm_plan_t plan, int32_t mode);

/* Programmatic dependent launch (default 1 = on): the GEMM kernel is launched
 * so that its set-up (barriers, tensor-memory allocation) may overlap the end
 * of the previous kernel in the stream; it waits for that kernel to complete
 * before reading or writing any global memory, so results never depend on
 * this setting.  0 launches with plain stream ordering.  GEMM_ERR_INVALID_ARG
 * for any other value.  No counterpart in the source pages (a launch detail). */
GEMM_API gemm_status_t gemm_plan_set_pdl(gemm_plan_t plan, int32_t enable);

/* How gemm_run would lay out this call: out[0] variant, out[1] CTAs launched,
 * out[2] units (CTAs or CTA pairs), out[3] tiles handed out whole, out[4]
 * units sharing the stream-K tail (0 = none), out[5] k-blocks in the tail.
 * Returns 0, or -1 on a rejected shape. */
GEMM_API int32_t gemm_plan_describe(gemm_plan_t plan, int64_t M, int64_t N, int64_t K,
                                    gemm_acc_t acc, int64_t out[6]);

/* Override the kernel variant chosen for a shape (-1 = automatic).  The
 * variants are listed by gemm_variant_name(0 .. gemm_variant_count()-1). */
GEMM_API gemm_status_t gemm_plan_set_variant(gemm_plan_t plan, int32_t variant);
GEMM_API int32_t gemm_variant_count(void);
GEMM_API const char* gemm_variant_name(int32_t variant);

/* Shape of a variant's unit of work: out[0] CTAs per unit (1, 2 or 4: a
 * CTA, a CTA pair, or a cluster of two pairs), out[1] x out[2] the
 * tile of C one unit owns (rows x columns), out[3] 1 if the MMA roles are
 * swapped (tiles then run over C's columns first).  Returns 0, or -1 for an
 * unknown variant. */
GEMM_API int32_t gemm_variant_info(int32_t variant, int32_t out[4]);

/* How many units of each kind fit on the plan's device at once: out[0]
 * SMs (one-CTA units), out[1] CTA pairs, out[2] clusters of two pairs
 * (each CTA takes one SM). */
GEMM_API gemm_status_t gemm_plan_resident_units(gemm_plan_t plan, int32_t out[3]);

/* The variant gemm_run would use for this shape and accumulation, and the
 * grid it would launch (CTAs), or -1 on a rejected shape. */
GEMM_API int32_t gemm_plan_pick_variant(gemm_plan_t plan, int64_t M, int64_t N, int64_t K,
                               gemm_acc_t acc, int32_t* grid_ctas);

/* Kernel launches issued through this plan so far (gemm_run and
 * gemm_run_host; the K == 0 zero-fill counts as one). */
GEMM_API uint64_t gemm_plan_launch_count(gemm_plan_t plan);

/* C = A x B^T for callers that cannot allocate device memory: no plan, and
 * no cudaMalloc, cudaFree or allocating library call anywhere in the call.
 * It always runs the one-CTA kernel (tc_single_128x256_s4) on whole tiles:
 * the same sum of the same products, but gemm_run may pick another tile
 * shape or split a tile's k-blocks over several SMs for the same shape, so
 * the two agree within the accumulation's tolerance, not bit for bit.  Who needs it: code running under an
 * allocator that owns all device memory (a framework's caching allocator or a
 * fixed arena, where a stray cudaMalloc can fail or fragment the pool), and
 * latency-bound loops that cannot afford cudaMalloc's implicit device
 * synchronisation.  The tutorial pages have no counterpart: this entry point
 * exists for those callers only.
 *
 * Arguments, layouts, shape and alignment rules, and the K == 0 / empty
 * cases are those of gemm_run; the device is the caller's current device,
 * and A, B and C must be device memory of that device (checked as in
 * gemm_run).
 * The kernel's only scratch (its 16-byte watchdog record) lives in a static
 * 256-byte device array inside the library, which every GPU that loads the
 * library holds until the process exits; a call whose scratch would not fit
 * is rejected with GEMM_ERR_INVALID_ARG (no current shape needs more than
 * 16 bytes).  The first call on each device does a one-time set-up (device
 * checks, kernel attributes, and the device address of the array via
 * cudaGetSymbolAddress), so make that first call before any stream capture.
 * Each call clears the record on `stream` before its launch.  All calls share
 * the one array: calls that overlap on the GPU race on it.  A watchdog
 * timeout cannot be reported by this asynchronous call: the kernel returns
 * early with C incomplete, and the next call clears the record; callers who
 * need the timeout report use gemm_run with a plan. */
GEMM_API gemm_status_t gemm_run_noalloc(const void* A, const void* B, void* C,
                                        int64_t M, int64_t N, int64_t K, gemm_acc_t acc,
                                        void* stream);

/* Human-readable name of a status code (static storage, never NULL). */
GEMM_API const char* gemm_status_string(gemm_status_t s);

/* Library version string (static storage). */
GEMM_API const char* gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GB300_GEMM_H_ */
