/*
 * qlin.h -- C ABI of libqlin: fused affine dequantise-into-matmul for
 * MLX-style packed 4/8-bit weights on NVIDIA GB300 (sm_103a).
 *
 * What the calls compute (the web pages the method comes from are cited by
 * title and section):
 *
 *   Packed weight format -- "epic: realize low-precision / quantized
 *   performance on the OpenXLA (IREE) backend", section Context: MLX 4/8-bit
 *   weights stay resident packed as a ui32 payload with one f16 (or, per
 *   "track(upstream-iree): fused dequant->matmul for the packed int8
 *   bandwidth win", section "What is already in-tree", bf16) scale and bias
 *   per group along K.
 *
 *   Reconstruction -- same section: bit-unpack, then w = q*scale + bias.
 *
 *   Fusion -- "track(upstream-iree): ...", section "The blocker (measured)":
 *   the matmul consumes the reconstructed weight; it is never written to DRAM.
 *
 *   M = 1 with N not a multiple of 4 -- "Metal backend: import qmv_impl from
 *   MLX": any N >= 1 is accepted.
 *
 * Shared notation and layouts (all row-major, all pointers are DEVICE
 * pointers owned by the caller; the library never allocates or frees):
 *
 *   bits        4 or 8; p = 32/bits codes per uint32 word
 *   group_size  64 (the only group size the kernels take; others return
 *               QLIN_ERR_UNSUPPORTED)
 *   W           N x K weights (output features x input features)
 *   wq          uint32 [N][K/p]; code k of row n sits at bits
 *               [bits*(k%p), bits*(k%p)+bits) of word wq[n][k/p]
 *               ("low bits first")
 *   scales,
 *   biases      sdtype [N][K/group_size]
 *   x           dtype [M][K]  (activations)
 *   y           dtype [M][N]  (y = x . W_hat^T, f32 accumulation, one
 *               round-to-nearest-even to dtype at the end)
 *
 * Errors: every call validates its arguments on the host before anything is
 * launched and returns a status; on failure nothing was launched and
 * qlin_last_error() (per calling thread) describes why.  The pages' own guards
 * likewise make unsupported settings fail fast instead of faulting mid-run
 * ("track(upstream-iree): ...", section "What is already in-tree").  A launch failure
 * reported by the CUDA runtime returns QLIN_ERR_CUDA.  Calls are asynchronous
 * on the given stream (a cudaStream_t passed as void*; NULL = legacy default
 * stream) and never synchronise the device.
 *
 * Device-side waits in the kernels are bounded; if one gives up it sets a
 * device status word that qlin_device_status() reads (and clears).
 */
#ifndef QLIN_H_
#define QLIN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QLIN_OK = 0,
  QLIN_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, K % group_size != 0, ... */
  QLIN_ERR_UNSUPPORTED = 2,  /* bits not in {4,8}, group_size != 64, dtype combination */
  QLIN_ERR_MISALIGNED = 3,   /* a pointer the 128-bit / TMA path needs 16-byte aligned is not */
  QLIN_ERR_CUDA = 4,         /* the CUDA runtime reported an error (see qlin_last_error) */
  QLIN_ERR_DEVICE_TIMEOUT = 5 /* a kernel's bounded wait gave up (qlin_device_status) */
} qlin_status;

typedef enum { QLIN_F32 = 0, QLIN_F16 = 1, QLIN_BF16 = 2 } qlin_dtype;

/* Human-readable name of a status code (static string).  No counterpart on
 * the pages: an addition of this library. */
const char* qlin_status_str(qlin_status s);

/* Detail of the last failing call made by this thread (static per-thread
 * buffer; empty string if none).  No counterpart on the pages: an addition of
 * this library, in the spirit of the guards that fail fast with a reason
 * ("track(upstream-iree): ...", section "What is already in-tree"). */
const char* qlin_last_error(void);

/* Library version as 10000*major + 100*minor + patch.  No counterpart on the
 * pages: an addition of this library. */
int qlin_version(void);

/*
 * Affine quantisation (load time; not on the per-token path).
 *   w       device float32 [N][K], finite values
 *   wq      device uint32 [N][K*bits/32]          (written)
 *   scales,
 *   biases  device sdtype [N][K/group_size]         (written)
 * Per row and group G of group_size consecutive k:
 *   scale = RNE_sdtype(fl32((max_G - min_G) / (2^bits - 1))),
 *   bias  = RNE_sdtype(min_G),
 *   q_k   = clamp(rint(fl32(fl32(w_k - bias) / scale)), 0, 2^bits - 1)
 *   (ties to even; q = 0 when the stored scale is 0).
 * The recipe is MLX's affine min/max quantisation with the rounding choices
 * spelled out (the pages give the format, not the quantiser).
 * sdtype: QLIN_F16 or QLIN_BF16.  Alignment: w and wq 16-byte aligned.
 */
qlin_status qlin_quantize_affine(const float* w, int64_t N, int64_t K, int bits, int group_size,
                                 qlin_dtype sdtype, uint32_t* wq, void* scales, void* biases,
                                 void* stream);

/*
 * Materialise the reconstruction w_hat[N][K] = RNE_out(q*scale + bias): one
 * correctly rounded step from the exact value, so it is bit-identical to a
 * host dequantisation (the pages require the in-graph reconstruction to match
 * the host dequant exactly: "track(upstream-iree): ...", section "What is
 * already in-tree").  out_dtype: QLIN_F32, or equal to
 * sdtype.  This is the unfused reference path and a test carrier; the matmul
 * entry points below never call it.  Alignment: wq and w_out 16-byte aligned.
 */
qlin_status qlin_dequant(const uint32_t* wq, const void* scales, const void* biases, int64_t N,
                         int64_t K, int bits, int group_size, qlin_dtype sdtype,
                         qlin_dtype out_dtype, void* w_out, void* stream);

/*
 * Fused matrix-vector / small-M product on CUDA cores (decode):
 *   y[m][n] = sum_k x[m][k] * (q[n][k]*scale[n][k/g] + bias[n][k/g])
 * for m < M, n < N.  dtype (QLIN_F16 or QLIN_BF16) is the type of x, y,
 * scales and biases.  Correct for any M >= 1 and N >= 1 (N need not be a
 * multiple of 4); fastest for M <= 4.  Alignment: x and wq 16-byte aligned.
 * Streams each packed word, scale and bias once per M-tile of 4 rows of x.
 * Defining passages: the reconstruction is consumed inside the product and
 * never written to DRAM ("track(upstream-iree): ...", section "The blocker
 * (measured)"); the M = 1 product for any N, including N not a multiple of 4
 * ("Metal backend: import qmv_impl from MLX").
 *
 * No workspace argument: the kernel gives each CTA whole rows and reduces
 * within a warp, so it needs no scratch memory, and the workspace pointer and
 * size query that a split-K design would need are not part of the call.
 */
qlin_status qlin_qmv(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                     void* y, int64_t M, int64_t N, int64_t K, int bits, int group_size,
                     qlin_dtype dtype, void* stream);

/*
 * Launch flags for the *_ex entry points.  No counterpart on the pages: an
 * addition of this library, aimed at the launch gaps between dependent
 * linears (the pages count ~678 dispatches per packed decode step: "epic:
 * realize low-precision / quantized performance on the OpenXLA (IREE)
 * backend", section "The measured fusion gate").
 *
 * QLIN_OVERLAP_PREVIOUS: launch as a programmatic dependent launch.  The
 *   kernel may start while the preceding kernel on the stream is still
 *   running and begins streaming its weights, scales and biases at once; it
 *   reads x and writes y only after that kernel has completed and its writes
 *   are visible.  The caller guarantees that the preceding work on the stream
 *   does not write wq, scales or biases (true for resident weights in a
 *   decode loop).  Hides launch and ramp-up time between dependent launches.
 */
#define QLIN_OVERLAP_PREVIOUS 1u

/* qlin_qmv with launch flags (0 = same as qlin_qmv).  Unknown flag bits
 * return QLIN_ERR_INVALID_ARG.  Product as qlin_qmv (same passages); the
 * flags are an addition of this library. */
qlin_status qlin_qmv_ex(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                        void* y, int64_t M, int64_t N, int64_t K, int bits, int group_size,
                        qlin_dtype dtype, unsigned flags, void* stream);

/*
 * A chain of dependent M = 1 products in one launch (a decode step).
 *
 * Link i computes y_i = x_i . W_hat_i^T with W_i given in the packed format
 * above (wq, scales, biases of shape [N][K]), where x_i is x0 (input = -1) or
 * the K elements starting at element input_offset of an earlier link's output
 * (0 <= input < i, input_offset + K <= N of that link).  The result is the
 * same as calling qlin_qmv on the links in order; the whole chain runs as one
 * persistent cooperative kernel whose CTAs stream every link's weights without
 * waiting and only wait, per link, until the row blocks of its input link are
 * complete.  The pages trace the packed path's slowness to unfused, separately
 * dispatched steps (~678 dispatches per decode step: "epic: realize
 * low-precision / quantized performance on the OpenXLA (IREE) backend",
 * section "The measured fusion gate").
 */
typedef struct {
  const uint32_t* wq;      /* [N][K*bits/32], 16-byte aligned */
  const void* scales;      /* dtype [N][K/group_size] */
  const void* biases;      /* dtype [N][K/group_size] */
  void* y;                 /* dtype [N] output; 16-byte aligned if a later link reads it */
  int64_t N, K;
  int32_t input;           /* -1: x0; else index of an earlier link */
  int32_t input_offset;    /* first element of that link's output read as x (x16 bytes aligned) */
} qlin_link;

/* Bytes of device scratch qlin_qmv_chain needs for n_links links (one 32-bit
 * completion counter per link, rounded up to 256 bytes).  No counterpart on
 * the pages: an addition of this library. */
size_t qlin_qmv_chain_workspace_size(int n_links);

/*
 * Run the chain.  x0: dtype [K of the links reading it], 16-byte aligned (may
 * be NULL when no link reads it).  workspace: device scratch of at least
 * qlin_qmv_chain_workspace_size(n_links) bytes, 16-byte aligned, owned by the
 * caller; the call zeroes it on the stream first, so concurrent chains need
 * separate workspaces.  1 <= n_links <= 160.  Outputs must not overlap any
 * weight or another link's output.  Errors as for qlin_qmv.
 */
qlin_status qlin_qmv_chain(const void* x0, const qlin_link* links, int n_links, int bits,
                           int group_size, qlin_dtype dtype, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * qlin_qmv_chain for callers that cannot allocate device memory (no
 * counterpart on the pages; an addition of this library).
 *
 * Same chain, same arguments and same results as qlin_qmv_chain, but the
 * per-link scratch counters live in a file-scope static device array inside
 * the library, so the call allocates nothing: for plugins whose host
 * framework owns all device memory through its own pool and forbids
 * cudaMalloc, and for deployments whose device memory budget is fixed at
 * start-up.  Limits: at most QLIN_CHAIN_STATIC_MAX_LINKS links (larger counts
 * return QLIN_ERR_INVALID_ARG); every GPU that loads the library keeps its
 * copy of the array until the process exits; all calls on a device share it
 * (each call zeroes the counters it uses on its stream first), so calls whose
 * kernels overlap on the GPU race and give wrong results.  The first call on
 * each device looks up the array's device address; make it before any stream
 * capture.
 */
#define QLIN_CHAIN_STATIC_MAX_LINKS 160
qlin_status qlin_qmv_chain_static(const void* x0, const qlin_link* links, int n_links, int bits,
                                  int group_size, qlin_dtype dtype, void* stream);

/*
 * The same product on the tensor cores (batched decode and prefill): packed
 * tiles are staged into shared memory by TMA, dequantised to dtype
 * (bit-identical to qlin_dequant's dtype output) into tensor memory as the
 * A operand of tcgen05 MMAs with f32 accumulators in tensor memory; when the
 * output has few tiles, K is split over a thread-block cluster and the
 * partial sums are added through distributed shared memory (no workspace).
 * Same arguments and result contract as qlin_qmv: for dtype QLIN_BF16 the
 * tensor-core operand carries w_hat as bf16 hi plus a bf16 residual lo (two
 * MMAs per K step), so rounding the operand to bf16 costs no accuracy.  Extra
 * requirement: K % 64 == 0 (always true for group 64) and x, wq 16-byte
 * aligned.  Defining passages: the target must fuse the dequantisation into
 * the matmul ("track(upstream-iree): ...", sections "The blocker (measured)"
 * and "Unblock criteria"), with bf16 scales and biases accepted (same page,
 * "What is already in-tree").
 */
qlin_status qlin_qmm(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                     void* y, int64_t M, int64_t N, int64_t K, int bits, int group_size,
                     qlin_dtype dtype, void* stream);

/* qlin_qmm with launch flags (0 = same as qlin_qmm).  QLIN_OVERLAP_PREVIOUS
 * as for qlin_qmv_ex: the launch and the kernel's set-up (barriers, tensor
 * memory, descriptor prefetch) overlap the preceding kernel on the stream; x
 * is read and y written only after that kernel has completed.  Unknown flag
 * bits return QLIN_ERR_INVALID_ARG.  Product as qlin_qmm (same passages); the
 * flags are an addition of this library. */
qlin_status qlin_qmm_ex(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                        void* y, int64_t M, int64_t N, int64_t K, int bits, int group_size,
                        qlin_dtype dtype, unsigned flags, void* stream);

/*
 * Dispatch to qlin_qmv when M < qlin_crossover_m_dtype(N, K, bits, dtype), else
 * qlin_qmm.
 * The product is the one both kernels define (same passages); choosing
 * between them by M is an addition of this library.
 */
qlin_status qlin_linear(const void* x, const uint32_t* wq, const void* scales,
                        const void* biases, void* y, int64_t M, int64_t N, int64_t K, int bits,
                        int group_size, qlin_dtype dtype, void* stream);

/* Smallest M for which qlin_linear picks the tensor-core path for activation
 * dtype `dtype`, from measurements on GB300: 4 for f16 when K > N; else 5
 * when N*K >= 6*2^20 and 9 below (qmv reads the weights once per 4 tokens).
 * `bits` does not change it (4- and 8-bit measured alike).  The environment
 * variable QLIN_CROSSOVER_M (read once per process) overrides it.  No
 * counterpart on the pages: an addition of this library. */
int64_t qlin_crossover_m_dtype(int64_t N, int64_t K, int bits, qlin_dtype dtype);

/* qlin_crossover_m_dtype for f16 activations. */
int64_t qlin_crossover_m(int64_t N, int64_t K, int bits);

/*
 * qlin_linear with a linear layer's epilogue:
 *
 *   y[m][n] = RNE_ydtype( sum_k x[m][k] * w_hat[n][k]  +  layer_bias[n] )
 *
 * layer_bias: dtype [N] (the activation dtype), added to the f32 accumulator
 *   before the single final rounding; NULL for no bias.  (This is the layer's
 *   own bias vector, not the quantisation biases of the packed format.)
 * y_dtype: QLIN_F32 (y is float [M][N], 4-byte aligned, no rounding) or the
 *   activation dtype (y as in qlin_linear).
 * The pages' ExecuTorch stack ships a 4-bit linear with bias ("Metal backend:
 * import qmv_impl from MLX", its stack of changes: "enable linear with bias",
 * "test 4-bit linear with bias"); the f32 output serves callers that keep the
 * residual stream in f32 (an addition of this library).
 *
 * Errors: as qlin_linear; y_dtype other than QLIN_F32 or dtype is
 * QLIN_ERR_UNSUPPORTED; layer_bias not 2-byte or an f32 y not 4-byte aligned
 * is QLIN_ERR_MISALIGNED.
 */
qlin_status qlin_linear_ex(const void* x, const uint32_t* wq, const void* scales,
                           const void* biases, const void* layer_bias, void* y, int64_t M,
                           int64_t N, int64_t K, int bits, int group_size, qlin_dtype dtype,
                           qlin_dtype y_dtype, void* stream);

/*
 * Read and clear the device status words of the current device (synchronises
 * the device).  *flags receives 0 when no kernel gave up a bounded wait since
 * the last call, else a bit mask of the waits that gave up (bits 0-7: the
 * tensor-core kernel, bits 8-15: the CUDA-core kernel, bits 16-23: the chain
 * kernel).  Returns QLIN_OK, or
 * QLIN_ERR_CUDA if the device could not be read.  No counterpart on the pages:
 * an addition of this library (a kernel that gives up a wait reports instead
 * of hanging, the device-side form of failing fast).
 */
qlin_status qlin_device_status(int* flags);

#ifdef __cplusplus
}
#endif

#endif /* QLIN_H_ */
