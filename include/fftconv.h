/*
 * fftconv — causal long convolution on one NVIDIA GB300 (sm_103a).
 *
 *   y[b,h,t] = sum_{j=0}^{t} u[b,h,j] * k[h,t-j],   t = 0..N-1
 *            = irfft(rfft(u[b,h,:], 2N) * rfft(k[h,:], 2N))[:N]
 *
 * (FlashFFTConv page, section 3.4 "The FFT Convolution and Its Hardware
 * Mismatch": the convolution, the convolution theorem and the zero-padding to
 * 2N for causal convolutions.)  The transform is computed as an order-p
 * Monarch decomposition (section 3.4 "The Monarch FFT Decomposition",
 * "Higher-order decompositions"): the length-N complex transform left after
 * the one-stage decimation in time (section 3.4 "The real-valued FFT
 * optimization") is factored into dense 16-, 32- and 64-point DFT
 * contractions on the tensor cores, with twiddle scaling and permutations
 * between them.  The kernel spectrum k_f is precomputed once per filter
 * (section 3.2, "Input and Kernel Preparation") and reused across the batch.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *   never frees them.  Each must be 16-byte aligned.
 * - u, y, w_in, w_out: contiguous [B][H][N] in the plan dtype (IEEE binary16
 *   for FFTCONV_F16, bfloat16 for FFTCONV_BF16).  k: contiguous float32
 *   [H][N].  k_f: opaque, fftconv_kf_bytes(plan, H) bytes, only valid for a
 *   plan with the same (N, dtype, order).
 * - y must not overlap any input (checked by address range).
 * - Work is enqueued on `stream` (cudaStream_t; NULL = legacy default stream)
 *   and the call returns without waiting.  Validation errors launch nothing.
 *   Asynchronous faults surface at the caller's next synchronisation.
 * - Results are bitwise deterministic for a given plan, inputs and GPU (no
 *   atomics in any reduction).
 * - B*H == 0 is valid and launches nothing.
 * - A plan is immutable after creation apart from its workspace; one plan may
 *   be used from several streams at once unless it needs a workspace
 *   (multi-pass lengths), in which case calls sharing it must be serialised.
 */
#ifndef FFTCONV_H
#define FFTCONV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fftconv_plan_s *fftconv_plan_t;
typedef void *fftconv_stream_t; /* a cudaStream_t */

typedef enum {
    FFTCONV_F16 = 0,  /* IEEE binary16 storage, fp16 tensor-core operands   */
    FFTCONV_BF16 = 1  /* bfloat16 storage, bf16 tensor-core operands        */
} fftconv_dtype_t;

typedef enum {
    FFTCONV_OK = 0,
    FFTCONV_ERR_INVALID = 1,     /* bad argument: NULL, overlap, negative size */
    FFTCONV_ERR_UNSUPPORTED = 2, /* length / order / dtype not supported       */
    FFTCONV_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned           */
    FFTCONV_ERR_WORKSPACE = 4,   /* multi-pass length without a big-enough workspace */
    FFTCONV_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed       */
    FFTCONV_ERR_ALLOC = 6,       /* device allocation failed                   */
    FFTCONV_ERR_TIMEOUT = 7      /* a bounded on-device wait gave up           */
} fftconv_status_t;

/* Which path a plan runs. */
typedef enum {
    FFTCONV_PATH_FUSED = 0,     /* one kernel, a whole row resident on chip        */
    FFTCONV_PATH_MULTIPASS = 1  /* outer stage through HBM, inner stages fused     */
} fftconv_path_t;

/* Host-side description of a plan (see fftconv_plan_query). */
typedef struct {
    int64_t N;            /* sequence length (real samples per row)              */
    int64_t M;            /* complex transform length after decimation, = N      */
    int32_t order;        /* p: number of Monarch factors                        */
    int32_t factors[8];   /* M = factors[0] * ... * factors[order-1], outer first */
    int32_t path;         /* fftconv_path_t                                      */
    int32_t dtype;        /* fftconv_dtype_t                                     */
    int64_t kf_bytes_per_channel; /* bytes of k_f per channel h                 */
    int64_t workspace_bytes_per_row; /* multi-pass workspace per (b,h) row; 0 if fused */
} fftconv_plan_info_t;

/*
 * Describe the plan that fftconv_plan_create would build, without touching
 * the GPU.  N must be a power of two with 2^10 <= N <= 2^21.  order = 0 picks
 * the factorization; a nonzero order is honoured or rejected.  Factorizations
 * (outer factor first; "Higher-order decompositions" of section 3.4):
 *   N = 4096, and 1024 / 2048 by default:
 *                         order 2, 64 x 64 (fused on the tensor cores; rows
 *                         of 1024 / 2048 zero-padded to 4096)
 *   N = 1024 / 2048 with order 3: N/256 x 16 x 16 (fused, warp-level MMAs)
 *   N = 8192, 16384, 32768: order 3, N/4096 x 64 x 64 (fused on the tensor
 *                         cores, the outer radix in registers); N = 32768
 *                         with order 4 runs multi-pass as below
 *   65536 <= N <= 2^19:   order 3, N/4096 x 64 x 64 (multi-pass; the default),
 *                         or order 4, N/16384 x 64 x 16 x 16, on request
 *   N >= 2^20:            order 4, N/2^18 x 64 x 64 x 64 (multi-pass; the
 *                         outer factor N/2^18 x 64 in one pass per direction)
 * Returns OK, INVALID (info NULL) or UNSUPPORTED.
 */
fftconv_status_t fftconv_plan_query(int64_t N, fftconv_dtype_t dtype, int order,
                                    fftconv_plan_info_t *info);

/*
 * Build a plan: choose the factorization (as fftconv_plan_query), build the
 * DFT-factor and twiddle tables in double precision, round them to the plan
 * dtype (twiddles stay float32), and upload them to the current device.
 * *out receives the plan; the plan owns its device tables until
 * fftconv_plan_destroy.  Returns OK, INVALID, UNSUPPORTED, ALLOC or CUDA.
 */
fftconv_status_t fftconv_plan_create(fftconv_plan_t *out, int64_t N, fftconv_dtype_t dtype,
                                     int order);

/*
 * Frequency-sparse plan (FlashFFTConv page, "Architectural Extensions:
 * Partial and Frequency-Sparse Convolutions", frequency-sparse part: a
 * structured subset of the bins of k_f is zeroed, chosen along the
 * decomposition so that whole blocks of work drop out).  As fftconv_plan_create, plus one band per
 * factor: band[0..nband-1], nband = the plan's order (query it first when
 * order = 0), outer factor first, each band >= 0.
 *
 * Pattern: the frequency index r = f mod N of spectrum bin f (0 <= f <= N of
 * the 2N-point spectrum of the real kernel) is written in mixed radix over
 * the factors, r = r_1 + M_1 r_2 + M_1 M_2 r_3 + ...; bin f is kept when
 * min(r_j, M_j - r_j) < band[j] for every j and set to zero otherwise (band
 * M_j/2 + 1 or more keeps axis j whole; band 0 drops every bin).  The forward
 * of such a plan computes
 *   y = first N outputs of IDFT_2N(DFT_2N(u0) . DFT_2N(k0) . m)
 * with m the 0/1 pattern on bins 0..N, mirrored to 2N - f (gated forms as
 * usual).  fftconv_kernel_fft and fftconv_kernel_fft_adjoint of the plan
 * zero the dropped bins of k_f; k_f is valid only for a plan with the same N,
 * dtype, order and band.
 *
 * Work skipped (multi-pass path): sub-row k0 of the inner transforms holds
 * the bins whose leading digits form k0; a pair of sub-rows (k0, R0 - k0)
 * whose bins are all dropped is not transformed, the first pass does not
 * write it and the last pass reads zeros in its place.  The fused
 * tensor-core kernel (N = 8192 .. 32768, outer factor R0 = N / 4096) works
 * on the same pairs inside one CTA: at R0 = 4 the pair (1, 3) is not run
 * when all its bins are dropped; R0 = 2 and 8 run every pair.  The other
 * fused paths apply the pattern through k_f only.
 *
 * fftconv_backward_dk and the partial and circular forwards return
 * UNSUPPORTED for a sparse plan.  Returns OK, INVALID (band NULL, nband not
 * the order, a negative band), UNSUPPORTED, ALLOC or CUDA.
 */
fftconv_status_t fftconv_plan_create_sparse(fftconv_plan_t *out, int64_t N, fftconv_dtype_t dtype,
                                            int order, const int32_t *band, int nband);

/*
 * Without touching the GPU: the pairs of sub-rows that a sparse plan with
 * these arguments would transform (*pairs_run) out of *pairs_total on the
 * multi-pass path and in the fused tensor-core kernel (N = 8192 .. 32768;
 * both 0 on the other fused paths).  Arguments as
 * fftconv_plan_create_sparse.  Returns OK, INVALID or UNSUPPORTED.
 */
fftconv_status_t fftconv_sparse_query(int64_t N, fftconv_dtype_t dtype, int order, const int32_t *band,
                                      int nband, int32_t *pairs_run, int32_t *pairs_total);

/*
 * The plan's bands (band[0..order-1]; band[order..7] = 0; a dense plan
 * reports M_j/2 + 1 for every axis) and the pairs of sub-rows that run
 * (*pairs_run) out of *pairs_total, as fftconv_sparse_query reports them.
 * Any output pointer may be NULL.  Returns OK or INVALID.
 */
fftconv_status_t fftconv_plan_get_band(fftconv_plan_t plan, int32_t *band, int32_t *pairs_run,
                                       int32_t *pairs_total);

/* Release a plan and its device tables (not the caller's buffers).  NULL is OK. */
fftconv_status_t fftconv_plan_destroy(fftconv_plan_t plan);

/* Copy the plan's description into *info. */
fftconv_status_t fftconv_plan_get_info(fftconv_plan_t plan, fftconv_plan_info_t *info);

/* Size in bytes of the k_f buffer for H channels (0 if plan is NULL). */
size_t fftconv_kf_bytes(fftconv_plan_t plan, int64_t H);

/*
 * Size in bytes of the device workspace a forward call over B*H rows needs:
 * 0 on the fused path; B*H*N*4 bytes (the 16-bit complex intermediate of
 * the outer stage) on the multi-pass path (section 3.4, "Kernel Fusion and
 * Recomputation Strategies": the outer layers spill to HBM).
 */
size_t fftconv_workspace_bytes(fftconv_plan_t plan, int64_t B, int64_t H);

/*
 * Attach a caller-owned device workspace (16-byte aligned) to the plan.
 * Passing NULL / 0 detaches it.  The plan does not free it.
 */
fftconv_status_t fftconv_set_workspace(fftconv_plan_t plan, void *dev_ptr, size_t bytes);

/*
 * Kernel spectrum: k_f[h] = the plan's encoding of rfft(k[h,:], 2N)
 * (section 3.2: the FFT of the filter, precomputed and reused across the
 * batch).  k is float32 [H][N] on the device; k_f is fftconv_kf_bytes(plan,H)
 * bytes on the device.  The encoding folds the decimation-in-time split and
 * merge (section 3.4, "The real-valued FFT optimization") into two complex
 * coefficients per frequency bin, stored in the plan dtype in the order the
 * forward kernel reads them.  The spectrum itself is computed in float32.
 * Allocates and frees stream-ordered temporary device memory (about
 * 16*H*N bytes).  Returns OK, INVALID, ALIGN, ALLOC or CUDA.
 */
fftconv_status_t fftconv_kernel_fft(fftconv_plan_t plan, const float *k, void *k_f, int64_t H,
                                    fftconv_stream_t stream);

/*
 * Forward causal convolution of B*H rows: y[b,h,:] = (u[b,h,:] * k[h,:])[0:N].
 * u, y: [B][H][N] plan dtype; k_f from fftconv_kernel_fft.  Arithmetic:
 * tensor-core contractions with 16-bit operands and float32 accumulation;
 * twiddle, decimation and gating products in float32; y rounded to the plan
 * dtype (nearest even).  Returns OK, INVALID, ALIGN, WORKSPACE or CUDA.
 */
fftconv_status_t fftconv_forward(fftconv_plan_t plan, const void *u, const void *k_f, void *y,
                                 int64_t B, int64_t H, fftconv_stream_t stream);

/*
 * Gated forward: y = w_out . ((u . w_in) * k) (section 3.4, "Gating
 * operation fusion": both gates applied inside the convolution kernel).
 * w_in, w_out: [B][H][N] plan dtype.  u . w_in is rounded to the plan dtype
 * before the first contraction; the output gate is applied in float32 before
 * the final rounding.  Same returns as fftconv_forward.
 */
fftconv_status_t fftconv_forward_gated(fftconv_plan_t plan, const void *u, const void *w_in,
                                       const void *w_out, const void *k_f, void *y, int64_t B,
                                       int64_t H, fftconv_stream_t stream);

/* Size of the library's own scratch array used by fftconv_forward_noalloc. */
#define FFTCONV_STATIC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * Forward convolution that allocates no device memory and takes no workspace.
 *
 * The FlashFFTConv page has no counterpart for this entry point.  It is for
 * callers that cannot call cudaMalloc themselves: code that runs inside a
 * host framework whose allocator owns every device byte, plug-ins that are
 * handed only their input and output buffers, and services that fix their
 * memory budget before they start.  Lengths above 16384 normally need the
 * caller's workspace of B*H*N*4 bytes (fftconv_set_workspace); this call
 * keeps that intermediate in one array of FFTCONV_STATIC_SCRATCH_BYTES
 * (64 MiB) compiled into the library, which every GPU that loads the
 * library reserves until the process exits.  Lengths up to 16384 use no
 * scratch at all and run the ordinary fused kernel.
 *
 * - Arguments, layouts, arithmetic and results are those of fftconv_forward.
 * - If B*H*N*4 exceeds FFTCONV_STATIC_SCRATCH_BYTES (for example more than
 *   64 rows of N = 262144, or more than 8 rows of N = 2^21), the call
 *   returns FFTCONV_ERR_WORKSPACE and launches nothing.
 * - The first call on a device looks up the array's address for the current
 *   device; make that first call before any stream capture on the device.
 *   The address is kept for the life of the process, so a device reset
 *   (cudaDeviceReset) after that first call is not supported: the array would
 *   live at a new address that the library does not look up again.
 * - Every call shares the one array.  Calls that can overlap on the GPU (on
 *   different streams or from different host threads) race and corrupt each
 *   other's results: serialise them.  Nothing in the array has to start at
 *   zero, since each call writes every word before it reads it.
 * - No cudaMalloc, cudaFree or other allocating routine is called.
 * Returns OK, INVALID, ALIGN, WORKSPACE or CUDA.
 */
fftconv_status_t fftconv_forward_noalloc(fftconv_plan_t plan, const void *u, const void *k_f, void *y,
                                         int64_t B, int64_t H, fftconv_stream_t stream);

/*
 * Forward convolution of rows that live in host memory: u (and w_in, w_out)
 * are copied to the device, convolved as fftconv_forward(_gated) would, and
 * y is copied back, all ordered on `stream`.  The rows are cut into chunks
 * (whole batch entries, or ranges of channels when B = 1) that pass through
 * three device buffer sets, so the copy of one chunk to the device, the
 * convolution of the one before and the copy back of the one before that
 * overlap (the plan keeps two internal copy streams for this, created on the
 * first call and released by fftconv_plan_destroy).  The FlashFFTConv page
 * has no counterpart: it assumes device-resident inputs; this call serves
 * callers whose sequences are produced and consumed on the host.
 *
 * - u, w_in, w_out, y: host memory, [B][H][N] in the plan dtype.  Page-locked
 *   memory (cudaHostAlloc / cudaHostRegister) is needed for the copies to
 *   overlap; pageable memory works but serialises them.  w_in and w_out are
 *   both NULL (plain convolution) or both non-NULL (gated).  y must not
 *   overlap the inputs.
 * - k_f: device, as for fftconv_forward.
 * - scratch: caller-owned device memory of at least
 *   fftconv_host_scratch_bytes(plan, B, H, gated) bytes, 16-byte aligned; it
 *   holds the three buffer sets and the multi-pass intermediate of one chunk,
 *   so no workspace needs to be attached.  It must not be used by anything
 *   else until the work on `stream` has completed.
 * - Returns OK, INVALID, ALIGN, WORKSPACE (scratch missing or too small) or
 *   CUDA.  When the call returns OK the copies and launches are queued; y is
 *   complete once `stream` has been synchronised.
 * - One plan must not run this call concurrently from two host threads.
 */
size_t fftconv_host_scratch_bytes(fftconv_plan_t plan, int64_t B, int64_t H, int gated);
fftconv_status_t fftconv_forward_host(fftconv_plan_t plan, const void *u, const void *w_in,
                                      const void *w_out, const void *k_f, void *y, int64_t B,
                                      int64_t H, void *scratch, size_t scratch_bytes,
                                      fftconv_stream_t stream);

/*
 * Backward pass (FlashFFTConv page, section 3.4, "Kernel Fusion and
 * Recomputation Strategies": the gradients with respect to u and k, with the
 * transforms recomputed rather than stored).  For y = conv(u, k) (causal, as
 * fftconv_forward) and an output gradient dy [B][H][N] in the plan dtype:
 *   du[b,h,j] = sum_{t=j}^{N-1} dy[b,h,t] k[h,t-j]              (correlation with k)
 *   dk[h,i]   = sum_b sum_{t=i}^{N-1} dy[b,h,t] u[b,h,t-i]       (batch sum of correlations with u)
 * and for the gated form y = w_out . conv(u . w_in, k):
 *   du = w_in . corr(w_out . dy, k),  dk[h] = sum_b corr(w_out . dy, u . w_in)
 * (the gate gradients, dw_in = u . corr(w_out . dy, k) and
 * dw_out = dy . conv(u . w_in, k), follow from du-style and forward calls).
 *
 * fftconv_kernel_fft_adjoint: as fftconv_kernel_fft, for conj(rfft(k, 2N));
 *   a forward call with this k_f computes the correlation with k.
 * fftconv_backward_du(_gated): du through the forward kernels with the
 *   adjoint k_f (the gated form swaps the gates); arguments, layouts,
 *   workspace and errors as fftconv_forward(_gated).
 * fftconv_backward_dk: dk float32 [H][N] on the device; w_in / w_out both
 *   NULL or both given; scratch: device memory of at least
 *   fftconv_backward_dk_scratch_bytes(plan, B, H) bytes (16-byte aligned; 0
 *   for 2N <= 8192, H*2N float32 complex values for 2N <= 65536, else
 *   (B + 1)*H*2N).  Computed in float32: the 2N-point transform of g + i x
 *   per row (g = w_out . dy, x = u . w_in), the per-channel sum over b of
 *   the cross spectra G conj X, one inverse transform per channel; for
 *   2N > 8192 as a four-step transform 2N = L1 x 2048 whose column
 *   transforms go through the scratch when 2N > 65536.  B = 0 writes zeros.
 *   Returns OK, INVALID, UNSUPPORTED (sparse or circular plan, too many
 *   rows), ALIGN, WORKSPACE or CUDA.
 */
fftconv_status_t fftconv_kernel_fft_adjoint(fftconv_plan_t plan, const float *k, void *k_f, int64_t H,
                                            fftconv_stream_t stream);
fftconv_status_t fftconv_backward_du(fftconv_plan_t plan, const void *dy, const void *k_f_adj, void *du,
                                     int64_t B, int64_t H, fftconv_stream_t stream);
fftconv_status_t fftconv_backward_du_gated(fftconv_plan_t plan, const void *dy, const void *w_in,
                                           const void *w_out, const void *k_f_adj, void *du, int64_t B,
                                           int64_t H, fftconv_stream_t stream);
size_t fftconv_backward_dk_scratch_bytes(fftconv_plan_t plan, int64_t B, int64_t H);
fftconv_status_t fftconv_backward_dk(fftconv_plan_t plan, const void *u, const void *dy, const void *w_in,
                                     const void *w_out, float *dk, int64_t B, int64_t H, void *scratch,
                                     size_t scratch_bytes, fftconv_stream_t stream);

/*
 * Partial convolution (FlashFFTConv page, "Architectural Extensions: Partial
 * and Frequency-Sparse Convolutions"): a kernel with at most C taps, where
 * C = W/2 and W is the plan's length, over sequences of any length N that is
 * a multiple of C (N may exceed 2^21):
 *   y[b,h,t] = sum_{j = max(0, t-C+1)}^{t} u[b,h,j] k[h,t-j]   (gated: w_out . conv(u . w_in, k))
 * k_f: fftconv_kernel_fft of the plan on k [H][W] whose taps at lags >= C
 * are zero (a shorter kernel, zero-padded).  The rows are cut into windows of
 * W inputs overlapping by C (window w covers inputs [(w-1)C, (w+1)C), zeros
 * before the start); each window is convolved by the plan's kernels and its
 * last C outputs are kept, so the convolution work per output is that of a
 * length-W transform.
 * - u, w_in, w_out, y: device, [B][H][N] in the plan dtype, 16-byte aligned;
 *   w_in, w_out both NULL or both given.
 * - scratch: device memory of fftconv_partial_scratch_bytes(plan, B, H, N,
 *   gated) bytes (the windowed inputs and outputs: two or four times the size
 *   of u, plus the multi-pass intermediate of the windows).
 * - Returns OK, INVALID, UNSUPPORTED (N not a multiple of C, or too many
 *   windowed rows), ALIGN, WORKSPACE or CUDA.
 */
size_t fftconv_partial_scratch_bytes(fftconv_plan_t plan, int64_t B, int64_t H, int64_t N, int gated);
fftconv_status_t fftconv_forward_partial(fftconv_plan_t plan, const void *u, const void *w_in,
                                         const void *w_out, const void *k_f, void *y, int64_t B, int64_t H,
                                         int64_t N, void *scratch, size_t scratch_bytes,
                                         fftconv_stream_t stream);

/*
 * Circular (non-causal) convolution of length C = W/2, W the plan's length
 * (the convolution theorem without zero padding or truncation):
 *   y[b,h,t] = sum_{j=0}^{C-1} u[b,h,j] k[h,(t-j) mod C]   (gated: w_out . conv(u . w_in, k))
 * k_f: fftconv_kernel_fft of the plan on k [H][W] holding the C taps followed
 * by C zeros.  Computed as outputs [C, 2C) of the plan's causal convolution of
 * [u, u] with [k, 0] (the first copy supplies the wrapped terms), i.e. one
 * window of fftconv_forward_partial whose first half wraps around.
 * u, w_in, w_out, y: device [B][H][C]; scratch: device memory of
 * fftconv_circular_scratch_bytes(plan, B, H, gated) bytes.  Errors as
 * fftconv_forward_partial.
 */
size_t fftconv_circular_scratch_bytes(fftconv_plan_t plan, int64_t B, int64_t H, int gated);
fftconv_status_t fftconv_forward_circular(fftconv_plan_t plan, const void *u, const void *w_in,
                                          const void *w_out, const void *k_f, void *y, int64_t B, int64_t H,
                                          void *scratch, size_t scratch_bytes, fftconv_stream_t stream);

/*
 * Native circular convolution of length C (FlashFFTConv page, section 5,
 * "Convolution Micro-Benchmarks": the non-causal FFT convolution, the
 * convolution theorem on C points without zero padding or truncation):
 *   y[b,h,t] = sum_{j=0}^{C-1} u[b,h,j] k[h,(t-j) mod C]   (gated: w_out . conv(u . w_in, k))
 * A circular plan transforms C real samples as M = C/2 complex points
 * (z[n] = u[2n] + i u[2n+1]), factored R0 x 64 x 64 with R0 = C/8192.
 * C = 16384 runs on the fused kernel (path FUSED, no workspace: both
 * 4096-point blocks of a row in shared memory); longer rows run multi-pass:
 * the first outer pass reads all R0 rows of z (no zero half) and the last
 * one writes all R0 output rows; the 4096-point sub-rows, the fold with the
 * kernel spectrum and the workspace are those of the multi-pass path.
 * - fftconv_circular_query: host only; C a power of two, 16384 <= C <= 2^19;
 *   info->N = C (samples per row), info->M = C/2, info->path FUSED for
 *   C = 16384, else MULTIPASS.  Returns OK, INVALID (info NULL) or
 *   UNSUPPORTED.
 * - fftconv_plan_create_circular: the plan (device tables on the current
 *   device).  On it, fftconv_kernel_fft and fftconv_kernel_fft_adjoint read
 *   k as [H][C] (all C taps of the circular kernel) and write k_f of
 *   fftconv_kf_bytes(plan, H) bytes; fftconv_forward and fftconv_forward_gated
 *   take u, w_in, w_out, y as device [B][H][C] and, on a multi-pass plan,
 *   a workspace of fftconv_workspace_bytes(plan, B, H) (= B H 2C) bytes
 *   (fftconv_set_workspace); fftconv_backward_du(_gated) with the adjoint
 *   k_f gives the input gradient (the circular correlation).  The partial,
 *   windowed-circular and kernel-gradient calls return UNSUPPORTED.
 *   Returns OK, INVALID, UNSUPPORTED, ALLOC or CUDA.
 */
fftconv_status_t fftconv_circular_query(int64_t C, fftconv_dtype_t dtype, fftconv_plan_info_t *info);
fftconv_status_t fftconv_plan_create_circular(fftconv_plan_t *out, int64_t C, fftconv_dtype_t dtype);

/*
 * Read and clear the plan's device error word (waits for `stream`).
 * *out = 0 if no bounded on-device wait has given up since the last call,
 * else FFTCONV_ERR_TIMEOUT.  Returns OK, INVALID or CUDA.
 */
fftconv_status_t fftconv_device_status(fftconv_plan_t plan, fftconv_stream_t stream, int *out);

/*
 * Failure-detection self-test: one CTA waits, with the same bounded waits the
 * kernels use (sleep != 0: the suspending form, at most about 2 s; else the
 * polling form), on an mbarrier phase that nothing completes.  The wait gives
 * up, records FFTCONV_ERR_TIMEOUT in the plan's error word (read it with
 * fftconv_device_status) and returns; the context stays usable.  Returns OK,
 * INVALID or CUDA.
 */
fftconv_status_t fftconv_selftest_wait(fftconv_plan_t plan, int sleep, fftconv_stream_t stream);

/* Static English text for a status code (never NULL). */
const char *fftconv_status_string(fftconv_status_t s);

/* Library version, e.g. "0.1.0". */
const char *fftconv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FFTCONV_H */
