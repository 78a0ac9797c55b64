/*
 * trellis.h — C ABI of the GB300 packed-Trellis decode and decode-and-multiply
 * library (libtrellis_gb300.so).
 *
 * The operation is the one computed by the `mlx_bun_trellis_wide_prefill`
 * Metal kernel on the page "mlx-bun 0.2.0 -> 0.4.0"
 * (package/src/model/trellis-wide-prefill.ts, kernel body and the
 * `wideTrellisPrefill` wrapper), and the dense "expand" decode named by
 * `expandTrellis` on the page "mlx-bun 0.4.0 -> 0.5.0"
 * (package/src/model/trellis-linear.ts).
 *
 * Data layout (all row-major, contiguous, caller-owned DEVICE memory):
 *   codes  uint32 [N, K*k/32]  Each row of K weights is cut into blocks of T
 *                              weights; a block is T*k/32 words whose bits,
 *                              lsb first, form one bit-string.  Weight t of a
 *                              block reads the L-bit window starting at bit
 *                              (T-1-t)*k of that bit-string, wrapping from the
 *                              block's last word to its word 0.
 *   scales bf16   [N]          one scale per output row.
 *   x      bf16   [M, K]       activations.
 *   out    bf16   [M, N] (trellis_gemm) or [N, K] (trellis_decode).
 * bf16 values travel as their 16-bit patterns (uint16_t).
 *
 * Per weight: win -> z = win*34038481 + 76625530 (mod 2^32) -> code = (sum of
 * the bytes of z) - 510 -> value = code / 147.800537109375 (fp32, correctly
 * rounded) -> w = bf16_rne(value * scale).  The product accumulates
 * float(w)*float(x) in fp32 and rounds each output once to bf16 (nearest even).
 *
 * Accepted geometry: T == 256, 1 <= k <= 8, k < L <= 24, K a positive
 * multiple of T, N >= 1, and for trellis_gemm 1 <= M <= 65536 (M <= 16 on the
 * CUDA cores, larger M on the tensor cores).  The page's wrapper accepts
 * k in {2, 3, 4} with L == 12; those geometries run on kernels specialised for
 * them, the rest on kernels that take the window width at run time (same
 * definition, same bits; slower).  Anything else returns
 * TRELLIS_ERR_UNSUPPORTED or TRELLIS_ERR_SHAPE before any launch.
 *
 * Every call is asynchronous on `stream` (0 = the legacy default stream): it
 * validates its arguments on the host, enqueues its kernels and returns
 * without synchronising.  Outputs are defined once the stream has been
 * synchronised.  A non-zero return means nothing was enqueued, except
 * TRELLIS_ERR_CUDA, which reports the CUDA error raised by the launch itself.
 * There is no CPU fallback.
 */
#ifndef TRELLIS_GB300_H
#define TRELLIS_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The library exports exactly the functions below; everything else in it has
 * hidden visibility (so that two copies of the library in one process never
 * share internal state). */
#if defined(__GNUC__) || defined(__clang__)
#define TRELLIS_API __attribute__((visibility("default")))
#else
#define TRELLIS_API
#endif

/* The CUDA runtime's stream handle, declared the way the runtime declares it,
 * so that this header does not need the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *cudaStream_t;

#define TRELLIS_ABI_VERSION 1

typedef enum trellis_status {
    TRELLIS_OK = 0,
    TRELLIS_ERR_NULL = -1,        /* a required pointer is NULL                        */
    TRELLIS_ERR_SHAPE = -2,       /* sizes inconsistent or out of range (K % T != 0)   */
    TRELLIS_ERR_UNSUPPORTED = -3, /* k, L, T or M outside the accepted set             */
    TRELLIS_ERR_ALIGN = -4,       /* a pointer misses its required alignment           */
    TRELLIS_ERR_CUDA = -5,        /* the CUDA runtime reported an error                */
    TRELLIS_ERR_TIMEOUT = -6,     /* a bounded device-side wait gave up                */
    TRELLIS_ERR_WORKSPACE = -7    /* workspace missing or smaller than required        */
} trellis_status;

/* ABI version compiled into the library (TRELLIS_ABI_VERSION). */
TRELLIS_API int trellis_abi_version(void);

/* Human-readable name of a status code; never NULL, static storage. */
TRELLIS_API const char *trellis_status_string(int status);

/*
 * trellis_decode — expand packed codes into the dense bf16 weight matrix
 * ("expand" mode of trellis-linear.ts on page "mlx-bun 0.4.0 -> 0.5.0"; the
 * arithmetic is the weight decode of the wide-prefill kernel body on page
 * "mlx-bun 0.2.0 -> 0.4.0").
 *
 *   codes   device, uint32 [N, K*k/32], 16-byte aligned.
 *   scales  device, bf16 [N], 2-byte aligned.
 *   out_bf16 device, bf16 [N, K], 16-byte aligned; fully overwritten.
 *   out[n, b*T + t] = bf16_rne(value(window_t(block b of row n)) * scales[n]).
 *
 * The result is bit-exact: every weight equals the definition above.
 * Errors: NULL pointer -> TRELLIS_ERR_NULL; misalignment -> TRELLIS_ERR_ALIGN;
 * K <= 0, N <= 0, K % T != 0 or N*K too large -> TRELLIS_ERR_SHAPE;
 * k, L or T outside the accepted set -> TRELLIS_ERR_UNSUPPORTED.
 */
TRELLIS_API int trellis_decode(const uint32_t *codes, const uint16_t *scales, int K, int N, int k, int L,
                               int T, uint16_t *out_bf16, cudaStream_t stream);

/*
 * trellis_gemm — fused decode-and-multiply out[m, n] = sum_k w[n, k] * x[m, k]
 * (the wide-prefill kernel of trellis-wide-prefill.ts, page "mlx-bun 0.2.0 ->
 * 0.4.0": each decoded weight row is shared by all M activation rows, partial
 * sums are fp32, each output is rounded once to bf16).
 *
 *   x       device, bf16 [M, K], 16-byte aligned (the page's wrapper also
 *           requires an aligned, row-contiguous x).
 *   codes   device, uint32 [N, K*k/32], 16-byte aligned.
 *   scales  device, bf16 [N].
 *   out     device, bf16 [M, N]; fully overwritten.
 *   1 <= M <= 65536.
 *
 * For M > 16 the decoded bf16 weight tiles are multiplied on the tensor cores
 * (tcgen05, fp32 accumulation in tensor memory): one launch serves up to 256
 * activation rows; larger M runs in 256-row launches, each decoding the
 * weights again (when M is not a multiple of 256 the last launch overlaps the
 * one before and rewrites those rows with the same bits).  That path needs no
 * workspace and its waits are bounded (see trellis_device_status).
 *
 * The summation order is fixed by the launch geometry, so repeated calls on
 * the same device give identical bits (the bits of trellis_gemm_ws).  For
 * M <= 16 the kernel balances work across all SMs by splitting rows' K-ranges
 * across CTAs; the split partial sums go through scratch memory.  trellis_gemm
 * takes that scratch from a fixed 4 MiB region of static device memory in the
 * library image (zero when loaded; every completed call leaves it ready for
 * the next).  The call itself never allocates and never synchronises: the
 * only host-side step is a one-time lookup of the region's address on each
 * device.  Under the CUDA runtime's default lazy module loading the driver
 * places the region and the kernels' code in device memory when a call first
 * needs them, and that load can wait for work in flight on the device; make
 * the first call per device (and bit width) before any stream capture and
 * before latency-sensitive work, or run with CUDA_MODULE_LOADING=EAGER, under
 * which the library's modules are loaded with it and even the first call
 * neither allocates nor waits.  All trellis_gemm calls on a device share the
 * region: calls that may overlap on the GPU (on two streams) race; use
 * trellis_gemm_ws with a workspace per stream for concurrent calls.
 * Errors: as trellis_decode, plus M outside 1..65536 -> TRELLIS_ERR_UNSUPPORTED;
 * on a device with more than 170 SMs the region is too small for some
 * M <= 16 shapes -> TRELLIS_ERR_WORKSPACE (use trellis_gemm_ws).
 */
TRELLIS_API int trellis_gemm(const uint16_t *x, const uint32_t *codes, const uint16_t *scales, int M, int K,
                             int N, int k, int L, int T, uint16_t *out, cudaStream_t stream);

/*
 * trellis_gemm_workspace_size — bytes of workspace trellis_gemm_ws needs for
 * this geometry on the CURRENT device (it depends on the SM count).
 * Writes the size to *bytes.  Same validation as trellis_gemm.
 */
TRELLIS_API int trellis_gemm_workspace_size(int M, int K, int N, int k, int L, int T, size_t *bytes);

/*
 * trellis_gemm_ws — trellis_gemm with a caller-owned workspace.
 *
 *   workspace        device, 256-byte aligned, at least the size reported by
 *                    trellis_gemm_workspace_size.
 *   workspace_bytes  its size in bytes.
 *
 * The workspace must be zero-filled before its first use.  Its first
 * 1 MiB holds per-tile counters that every completed call leaves at zero; the
 * rest holds partial sums that need no clearing, so the workspace can be
 * reused, for any geometry that fits it, without clearing.  Geometries with
 * more than 2^18 row tiles (tiles are 64 rows) are rejected with
 * TRELLIS_ERR_SHAPE.  Two calls that may overlap on the GPU must not
 * share a workspace.  A workspace sized for one geometry serves any geometry
 * whose reported size is not larger.
 * Errors: as trellis_gemm, plus TRELLIS_ERR_WORKSPACE when the workspace is
 * NULL or too small, TRELLIS_ERR_ALIGN when it is misaligned.
 */
TRELLIS_API int trellis_gemm_ws(const uint16_t *x, const uint32_t *codes, const uint16_t *scales, int M,
                                int K, int N, int k, int L, int T, uint16_t *out, void *workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * trellis_device_status — synchronise `stream`, then report whether a bounded
 * device-side wait of the tensor-core product gave up since the last query
 * (TRELLIS_ERR_TIMEOUT; the affected outputs are undefined) or not
 * (TRELLIS_OK).  Clears the flag.  A wait gives up after 2 s of wall-clock
 * time; the kernel then waits (bounded the same way) for its own copies and
 * tensor-core operations still in flight, releases its tensor memory and
 * returns, so the context stays usable.  The flag is one word per device,
 * shared by every stream and every caller on that device: a timeout on any
 * stream is reported to, and cleared by, whichever query comes first, and
 * synchronising `stream` does not wait for work on other streams.
 * No counterpart on the pages: it is how the library surfaces its own wait
 * limits.
 */
TRELLIS_API int trellis_device_status(cudaStream_t stream);

/*
 * trellis_selftest_wait_timeout — enqueue on `stream` a one-thread kernel
 * whose bounded wait (50 ms) runs out because nothing arrives on its barrier;
 * it sets the same device error word as a product wait that gives up, so the
 * next trellis_device_status returns TRELLIS_ERR_TIMEOUT.  Checks the failure
 * reporting path without a hang or a fault.  Returns TRELLIS_OK or
 * TRELLIS_ERR_CUDA.
 */
TRELLIS_API int trellis_selftest_wait_timeout(cudaStream_t stream);

/*
 * trellis_gemm_gateup — the two projections of a gated MLP that share x, in
 * one pass over x: out_gate = x * W_gate^T and out_up = x * W_up^T (each as
 * trellis_gemm computes it, the same bits as two trellis_gemm calls up to the
 * split-K summation order), and, when out_act is not NULL,
 * out_act = bf16(silu(out_gate) * out_up) elementwise with
 * silu(v) = v / (1 + e^-v) evaluated in fp32 from the bf16 outputs.  The
 * fused gate/up kernels are named on the page "mlx-bun 0.4.0 -> 0.5.0" without
 * their bodies; this is the plainest reading (two trellis products sharing x,
 * an optional SiLU-gated product).
 *
 *   codes_gate/scales_gate, codes_up/scales_up: two weight matrices [N, K], as
 *           for trellis_gemm (same k, K, N).
 *   out_gate, out_up: device, bf16 [M, N]; out_act: bf16 [M, N] or NULL.
 *   workspace: as trellis_gemm_ws, sized by trellis_gemm_gateup_workspace_size
 *           (0 bytes for M > 16).
 * For M <= 16 with k in {2,3,4} and L == 12, both matrices' rows are decoded
 * in one launch (the activations are staged once); other geometries run two
 * launches through the one workspace; for M > 16 each matrix takes the
 * tensor-core path.
 * Errors: as trellis_gemm_ws for either matrix; out_act misaligned ->
 * TRELLIS_ERR_ALIGN.
 */
TRELLIS_API int trellis_gemm_gateup(const uint16_t *x, const uint32_t *codes_gate, const uint16_t *scales_gate,
                                    const uint32_t *codes_up, const uint16_t *scales_up, int M, int K, int N, int k,
                                    int L, int T, uint16_t *out_gate, uint16_t *out_up, uint16_t *out_act,
                                    void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * trellis_gemm_gateup_workspace_size — bytes of workspace trellis_gemm_gateup
 * needs on the current device.  Same validation as trellis_gemm.
 */
TRELLIS_API int trellis_gemm_gateup_workspace_size(int M, int K, int N, int k, int L, int T, size_t *bytes);

/*
 * trellis_gemm_noalloc — trellis_gemm for callers that cannot allocate device
 * memory.  The pages have no counterpart: this is a library convenience.
 *
 * Same arguments, validation, arithmetic and results as trellis_gemm, but the
 * scratch memory of the split-K reduction comes from a fixed 16 MiB array that
 * the library holds on every GPU that loads it, until the process exits.  It
 * never calls cudaMalloc, cudaFree or any allocating routine, so it suits code
 * that must not allocate: allocator or memory-pool callbacks, processes that
 * reserve all device memory up front, runtimes that forbid allocation on the
 * hot path.
 *
 * The first call on each device does a one-time set-up with that device
 * current (it looks up the array's device address and clears its counter
 * region, synchronising the device).  Under the CUDA runtime's default lazy
 * module loading, the array and the kernels' code are placed in device memory
 * when that first call touches them, not when the library is loaded: a
 * process that reserves all
 * free device memory up front must make its first call (per device and per
 * bit width k, whose kernels are separate modules) before reserving, or run
 * with CUDA_MODULE_LOADING=EAGER.  Every call shares the array: calls that may
 * overlap on the same GPU (for instance on two streams) race and must be
 * serialised by the caller.  Same argument checks, in the same order, as
 * trellis_gemm; then geometries whose scratch (as reported by
 * trellis_gemm_workspace_size) exceeds 16 MiB are rejected with
 * TRELLIS_ERR_WORKSPACE before any launch (a guard for devices with more than
 * 853 SMs: below that the scratch of every accepted geometry fits).
 */
TRELLIS_API int trellis_gemm_noalloc(const uint16_t *x, const uint32_t *codes, const uint16_t *scales, int M,
                                     int K, int N, int k, int L, int T, uint16_t *out, cudaStream_t stream);

/*
 * trellis_gemm_packed — token packing: several independent groups of
 * activation rows (sequences) multiplied by the same weights in ONE product,
 * as `mapPackedTokens` on the page "mlx-bun 0.4.0 -> 0.5.0" (token-groups.ts)
 * packs the real tokens of several sequences for a tokenwise operation and
 * restores each group's rows afterwards.  Packing raises the M the product
 * sees, so the weights are decoded once for all groups instead of once per
 * group.
 *
 *   xs      HOST array of `groups` device pointers; xs[g] is bf16 [rows[g], K],
 *           16-byte aligned.
 *   rows    HOST array of `groups` row counts, each >= 1; M = sum(rows) must
 *           be in 1..65536.
 *   codes, scales, K, N, k, L, T: as trellis_gemm.
 *   outs    HOST array of `groups` device pointers; outs[g] is bf16
 *           [rows[g], N], 2-byte aligned; fully overwritten.
 *   workspace, workspace_bytes: device, 256-byte aligned, zero-filled before
 *           its first use, at least trellis_gemm_packed_workspace_size bytes;
 *           it holds the packed x [M, K], the packed output [M, N] and the
 *           product's own workspace.
 *
 * outs[g] equals rows pos_g .. pos_g + rows[g] - 1 of trellis_gemm on the
 * concatenation of the xs (pos_g = rows of the groups before g): the groups are
 * gathered by one copy kernel (per 64 groups), multiplied once and scattered
 * back by one more, all on `stream`.  One group is multiplied in place (no
 * copies), as on the page.
 * Errors: groups < 1 or a NULL array or pointer -> TRELLIS_ERR_NULL or
 * TRELLIS_ERR_SHAPE (rows[g] < 1); M outside 1..65536 ->
 * TRELLIS_ERR_UNSUPPORTED; the rest as trellis_gemm_ws.  All checks run before
 * anything is enqueued.
 */
TRELLIS_API int trellis_gemm_packed(const uint16_t *const *xs, const int *rows, int groups, const uint32_t *codes,
                                    const uint16_t *scales, int K, int N, int k, int L, int T, uint16_t *const *outs,
                                    void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * trellis_gemm_packed_workspace_size — bytes of workspace trellis_gemm_packed
 * needs for these groups on the current device.  Same validation as
 * trellis_gemm_packed for the sizes.
 */
TRELLIS_API int trellis_gemm_packed_workspace_size(const int *rows, int groups, int K, int N, int k, int L, int T,
                                                   size_t *bytes);

#ifdef __cplusplus
}
#endif

#endif /* TRELLIS_GB300_H */
