/*
 * dsc.h -- C ABI of the B300 (sm_103a) Dynamic Short Convolution library,
 * libdsc.so.
 *
 * The operation (from "Technische Samenvatting: Dynamische Korte Convoluties
 * Verbeteren Transformers", Methodologie: Mechanisme, Parametrisatie,
 * Plaatsing; and "Dynamic Short Convolutions: The 'Locality Bias'
 * Transformers Were Missing", Methodology, section 1):
 *
 *   y[b,t,c] = residual * x[b,t,c] + sum_{k=0}^{W-1} w[b,t,g(c),k] * x[b,t-k,c]
 *
 * with x[b,t-k,c] = 0 for t-k < 0 (zero padding per sequence b, no carried
 * state), g(c) = floor(c / H) (one filter shared by H consecutive channels)
 * and G = C / H filters per token.  In the low-rank parameterisation the
 * filters are w[b,t,g,k] = sum_r z[b,t,r] * U[r, g*W + k]; they are formed
 * on-chip and never written to memory (same summary, Efficiente
 * Trainingsimplementatie: Fused Low-Rank Kernel).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  Every tensor argument is a pointer to DEVICE memory, dense and
 * row-major (last index fastest), owned by the caller:
 *     x, y, dy, dx : [B, T, C]
 *     w, dw        : [B, T, G, W]            (tap k fastest)
 *     z, dz        : [B, T, R]
 *     U, dU        : [R, G*W]                (column j = g*W + k)
 * The library never allocates, frees or synchronises.  Outputs are
 * overwritten, never accumulated into.  Outputs may not alias inputs.
 * Element type.  All tensors of one call share `dtype`: DSC_F32 (fp32) or
 * DSC_BF16 (bfloat16).  Arithmetic is fp32; a bf16 result is rounded to
 * nearest-even once, after the fp32 sum (the residual included).
 * Ordering.  Work is enqueued on `stream` (a cudaStream_t; NULL = the
 * legacy default stream) and runs asynchronously; the call returns once it
 * is enqueued.
 * Shapes.  B >= 0, T >= 0 (B*T == 0 is a no-op), C >= 1, H >= 1, C % H == 0,
 * 1 <= W <= 4 (W > 4 gives DSC_ERR_UNSUPPORTED).  C must be a multiple of 8
 * (bf16) or 4 (fp32), and every pointer 16-byte aligned, else
 * DSC_ERR_ALIGNMENT.  Any T is accepted, including T < W.
 * Errors.  Arguments are validated on the host before anything is
 * enqueued; a failed check returns its status and enqueues nothing.  A CUDA
 * launch failure returns DSC_ERR_CUDA.  The library never aborts, traps or
 * asserts.
 */
#ifndef DSC_H_
#define DSC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSC_OK = 0,
  DSC_ERR_INVALID_ARG = 1, /* null pointer, negative size, C % H != 0, ...  */
  DSC_ERR_ALIGNMENT = 2,   /* pointer not 16-byte aligned, C not a multiple */
  DSC_ERR_UNSUPPORTED = 3, /* valid but not built: W > 4, R > 32, ...       */
  DSC_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required    */
  DSC_ERR_CUDA = 5         /* a CUDA call failed (launch error)             */
} dsc_status_t;

typedef enum { DSC_F32 = 0, DSC_BF16 = 1 } dsc_dtype_t;

/* Version of this ABI (bumped on any incompatible change). */
int dsc_abi_version(void);

/* Static name of a status code. */
const char* dsc_status_string(dsc_status_t status);

/*
 * Head-wise DSC forward (Mechanisme + Parametrisatie item 2 + Plaatsing).
 *   in : x [B,T,C], w [B,T,C/H,W]
 *   out: y [B,T,C] = residual*x + sum_k w[.,t,g(c),k] * x[.,t-k,c]
 * `residual` != 0 adds x (the X = X + DSC(X) placement).
 */
dsc_status_t dsc_headwise_fwd(const void* x, const void* w, void* y,
                              int64_t B, int64_t T, int64_t C, int64_t H,
                              int64_t W, int residual, dsc_dtype_t dtype,
                              void* stream);

/*
 * Head-wise DSC backward: the chain rule of dsc_headwise_fwd (the pages
 * state no backward formula; this one is derived from the forward).
 *   in : x [B,T,C], w [B,T,G,W], dy [B,T,C] (gradient of the loss wrt y)
 *   out: dx [B,T,C]:   dx[b,s,c] = residual*dy[b,s,c]
 *                                 + sum_{k: s+k<T} w[b,s+k,g(c),k] dy[b,s+k,c]
 *        dw [B,T,G,W]: dw[b,t,g,k] = sum_{c=gH}^{gH+H-1} dy[b,t,c] x[b,t-k,c]
 *                                    (0 for t-k < 0)
 */
dsc_status_t dsc_headwise_bwd(const void* x, const void* w, const void* dy,
                              void* dx, void* dw, int64_t B, int64_t T,
                              int64_t C, int64_t H, int64_t W, int residual,
                              dsc_dtype_t dtype, void* stream);

/*
 * Low-rank fused DSC forward (Parametrisatie item 1; Fused Low-Rank Kernel):
 * the filters w[b,t,g,k] = sum_r z[b,t,r] U[r,g*W+k] are generated on-chip
 * in fp32 (never rounded, never stored) and applied at once.
 *   in : x [B,T,C], z [B,T,R], U [R,G*W]
 *   out: y [B,T,C]
 * 1 <= R <= 32.  H = 1 and power-of-two H up to 32 are built; other H give
 * DSC_ERR_UNSUPPORTED.
 */
dsc_status_t dsc_lowrank_fwd(const void* x, const void* z, const void* U,
                             void* y, int64_t B, int64_t T, int64_t C,
                             int64_t H, int64_t W, int64_t R, int residual,
                             dsc_dtype_t dtype, void* stream);

/*
 * Bytes of device workspace dsc_lowrank_bwd needs for these arguments
 * (deterministic fp32 partial sums of dz and dU).  0 for an empty problem
 * or unsupported arguments.
 */
size_t dsc_lowrank_bwd_workspace_size(int64_t B, int64_t T, int64_t C,
                                      int64_t H, int64_t W, int64_t R,
                                      dsc_dtype_t dtype);

/*
 * Low-rank fused DSC backward: the chain rule of dsc_lowrank_fwd.
 *   in : x [B,T,C], z [B,T,R], U [R,G*W], dy [B,T,C]
 *   out: dx [B,T,C]  (as dsc_headwise_bwd, with the generated filters)
 *        dz [B,T,R]: dz[b,t,r] = sum_j dw[b,t,j] U[r,j]
 *        dU [R,G*W]: dU[r,j]   = sum_{b,t} z[b,t,r] dw[b,t,j]
 *   where dw is the head-wise filter gradient, kept on-chip in fp32.
 * workspace: caller-owned device memory of at least
 * dsc_lowrank_bwd_workspace_size(...) bytes, 16-byte aligned; its contents
 * on entry do not matter and are clobbered.  Partial sums are combined in a
 * fixed order, so results are bitwise reproducible run to run.
 */
dsc_status_t dsc_lowrank_bwd(const void* x, const void* z, const void* U,
                             const void* dy, void* dx, void* dz, void* dU,
                             void* workspace, size_t workspace_bytes,
                             int64_t B, int64_t T, int64_t C, int64_t H,
                             int64_t W, int64_t R, int residual,
                             dsc_dtype_t dtype, void* stream);

/*
 * Static short convolution: the special case of DSC whose filters do not
 * depend on the token ("Dynamic Short Convolutions: The 'Locality Bias'
 * Transformers Were Missing", Methodology: Adaptive Filtering at Scale,
 * 1. Mathematical Intuition, the standard convolution; the static kernels of
 * its Figure 1 compute the same operation).  One filter per channel:
 *   y[b,t,c] = residual*x[b,t,c] + sum_{k=0}^{W-1} w[c,k] x[b,t-k,c]
 * with x = 0 before t = 0 of each sequence (k = 0 is the current token).
 *   x, y : [B, T, C]     w : [C, W]
 * Equal to dsc_headwise_fwd with H = 1 and w broadcast over b and t.
 * Arithmetic fp32, y rounded once.  Shape, alignment and aliasing rules as
 * for dsc_headwise_fwd; B*T = 0 is a no-op.
 */
dsc_status_t dsc_static_fwd(const void* x, const void* w, void* y, int64_t B,
                            int64_t T, int64_t C, int64_t W, int residual,
                            dsc_dtype_t dtype, void* stream);

/* Bytes of device workspace dsc_static_bwd needs for this shape (a function
 * of the shape only); 0 for an invalid shape or B*T = 0. */
size_t dsc_static_bwd_workspace_size(int64_t B, int64_t T, int64_t C,
                                     int64_t W, dsc_dtype_t dtype);

/*
 * Backward of dsc_static_fwd:
 *   dx[b,s,c] = residual*dy[b,s,c] + sum_{k: s+k<T} w[c,k] dy[b,s+k,c]
 *   dw[c,k]   = sum_{b,t>=k} dy[b,t,c] x[b,t-k,c]      (over every token)
 * dw is accumulated in fp32 (one partial per token range in the workspace,
 * then added in a fixed order: bitwise reproducible) and rounded once.
 * workspace: caller-owned device memory of at least
 * dsc_static_bwd_workspace_size(...) bytes, 16-byte aligned, clobbered.
 * B*T = 0 writes zeros to dw and touches nothing else (x, w, dy, dx and the
 * workspace may then be NULL).
 */
dsc_status_t dsc_static_bwd(const void* x, const void* w, const void* dy,
                            void* dx, void* dw, void* workspace,
                            size_t workspace_bytes, int64_t B, int64_t T,
                            int64_t C, int64_t W, int residual,
                            dsc_dtype_t dtype, void* stream);

/*
 * Decode step (inference, one new token per sequence) with a carried state.
 * The pages leave inference to future engineering; this is the forward
 * definition evaluated at one new position t with the last W-1 inputs of
 * each sequence kept as state:
 *   y[b,c]        = residual*x[b,c] + w[b,g(c),0] x[b,c]
 *                   + sum_{k=1}^{W-1} w[b,g(c),k] state[b,k-1,c]
 *   state[b,0,c] <- x[b,c],  state[b,j,c] <- state[b,j-1,c]   (j >= 1)
 * where state[b,j] holds the input at time t-1-j (all zeros at the start of
 * a sequence, the causal zero padding).
 *   x, y  : [B, C]          w : [B, C/H, W]
 *   state : [B, W-1, C], read and updated in place (may be NULL when W = 1)
 * Same element type for all; arithmetic fp32, y rounded once; the state
 * keeps exact copies of the inputs.  y may not alias x, state may not alias
 * x or y.  Alignment, shape and error rules as for the other entry points
 * (T is 1); B = 0 is a no-op.
 */
dsc_status_t dsc_headwise_decode(const void* x, const void* w, void* state, void* y,
                                 int64_t B, int64_t C, int64_t H, int64_t W, int residual,
                                 dsc_dtype_t dtype, void* stream);

/*
 * Low-rank decode step: the taps w[b,g,k] = sum_r z[b,r] U[r,g*W+k] are
 * formed in fp32 (never rounded), then the step above.  z : [B, R],
 * U : [R, (C/H)*W], 1 <= R <= 32.
 */
dsc_status_t dsc_lowrank_decode(const void* x, const void* z, const void* U, void* state,
                                void* y, int64_t B, int64_t C, int64_t H, int64_t W, int64_t R,
                                int residual, dsc_dtype_t dtype, void* stream);

/*
 * Decode step merged with the projection that produces its input
 * ("Dynamic Short Convolutions: The 'Locality Bias' Transformers Were
 * Missing", Limitations: for inference the convolution is to be merged into
 * the matmul that precedes it).  The step's input is computed in the same
 * kernel as
 *   x[b,c] = sum_{d<D} h[b,d] Wp[c,d]        (fp32 accumulation)
 * rounded once to the I/O type (the value a separate projection would
 * store), then the decode step of dsc_headwise_decode runs on it: y and the
 * state are exactly what that projection followed by dsc_headwise_decode
 * produce, up to the summation order of x.  x itself is not written; with
 * W > 1 it is row 0 of the updated state.
 *   h : [B, D] hidden states of the new tokens    Wp : [C, D] (a linear
 *   layer's weight: out_features x in_features)   w : [B, C/H, W]
 *   state : [B, W-1, C], read and updated in place (may be NULL when W = 1)
 *   y : [B, C]
 * Same element type for all.  1 <= D <= 2^24 with 16-byte rows (D a
 * multiple of 8 for bf16, 4 for fp32, else DSC_ERR_ALIGNMENT); B <= 2^24.
 * y may not alias h or Wp; the state may not alias h, Wp or y.  Other rules
 * as for dsc_headwise_decode; B = 0 is a no-op.  The kernel streams Wp once
 * per block of 8 sequences (later blocks from L2), so it is built for
 * decode batches; it is not a general GEMM.
 */
dsc_status_t dsc_headwise_proj_decode(const void* h, const void* Wp, const void* w,
                                      void* state, void* y, int64_t B, int64_t D,
                                      int64_t C, int64_t H, int64_t W, int residual,
                                      dsc_dtype_t dtype, void* stream);

/*
 * The same for the low-rank parameterisation: the projection as above,
 * then the step of dsc_lowrank_decode (taps sum_r z[b,r] U[r,g*W+k] in fp32).
 * z : [B, R], U : [R, (C/H)*W], 1 <= R <= 32.
 */
dsc_status_t dsc_lowrank_proj_decode(const void* h, const void* Wp, const void* z,
                                     const void* U, void* state, void* y, int64_t B,
                                     int64_t D, int64_t C, int64_t H, int64_t W, int64_t R,
                                     int residual, dsc_dtype_t dtype, void* stream);

/*
 * Which low-rank kernels these arguments run on: bit 0 set if
 * dsc_lowrank_fwd uses the tensor cores (tcgen05: bf16, R in {8, 16, 24,
 * 32}, 1 <= W <= 4, H = 1, or H > 1 with (64/H)*W and (C/H)*W multiples of
 * 8), bit 1 set if dsc_lowrank_bwd does (bf16, R in {8, 16, 24, 32},
 * 1 <= W <= 4, any H); a clear bit means the CUDA-core kernels.  -1 if the
 * arguments are invalid or unsupported.  Host only; touches no device.
 */
int dsc_lowrank_uses_tensor_cores(int64_t B, int64_t T, int64_t C, int64_t H,
                                  int64_t W, int64_t R, dsc_dtype_t dtype);

/*
 * Which head-wise kernels these arguments run on: bit 0 set if
 * dsc_headwise_fwd uses the TMA-staged kernel, bit 1 set if
 * dsc_headwise_bwd does; a clear bit means the register-streaming kernels.
 * The TMA kernels take bf16 with (H, W) whose filter rows make a 16-byte
 * multiple box: items of 64 channels for H = 8 (any W), (16, 2), (16, 4),
 * (32, 4) and the backward of (16, 3) and (64, 4) (whose filter rows are
 * loaded as a wider aligned box; C a multiple of 128), and of 128 channels
 * for (16, 1), the forward of (16, 3) and (64, 4), and (32, 2); C must be a
 * multiple of the item width.  -1 if the arguments are invalid.  Host only;
 * touches no device.
 */
int dsc_headwise_uses_tma(int64_t B, int64_t T, int64_t C, int64_t H, int64_t W,
                          dsc_dtype_t dtype);

/*
 * Diagnostic: the device error word of the tensor-core and TMA kernels on
 * the current device.  0 means no error; otherwise it holds the code of the
 * first bounded wait that gave up (1 producer, 2 MMA issuer, 3 epilogue,
 * 4 store, 5 second MMA issuer), after which that kernel returned early and
 * its outputs are
 * invalid.  `reset` != 0 clears the word.  Synchronous (it copies one word
 * from the device); not meant for the hot path.
 */
dsc_status_t dsc_device_error(unsigned int* code, int reset);

/*
 * Self-tests of the failure path of the tensor-core low-rank kernels
 * (diagnostic; not for the hot path).  Every wait of those kernels on an
 * mbarrier is bounded: after a time limit it gives up, records a code in the
 * device error word (dsc_device_error), lets the CTA's copies and MMAs in
 * flight finish, frees the CTA's TMEM and returns, so a broken pipeline
 * ends with an error status instead of hanging the GPU.  These entry points
 * run dsc_lowrank_fwd / dsc_lowrank_bwd with every limit set to
 * wait_limit_ns (1 us .. 1 s; the normal limit is 1 s) and with a producer
 * that issues no loads, so the waits of the other roles run out.  Expected
 * result: the call enqueues and returns DSC_OK, the kernels end within a
 * few limits, dsc_device_error then reports a nonzero code (2, 3 or 5), the
 * outputs are unspecified, and the next normal call on the device runs
 * correctly.  Arguments as for dsc_lowrank_fwd / dsc_lowrank_bwd, plus
 * wait_limit_ns; DSC_ERR_UNSUPPORTED when the arguments do not take the
 * tensor-core path (dsc_lowrank_uses_tensor_cores), DSC_ERR_INVALID_ARG
 * for an empty problem or a limit outside the range.  Nothing faults or
 * traps: the waits simply run out.
 */
dsc_status_t dsc_lowrank_fwd_selftest_timeout(const void* x, const void* z,
                                              const void* U, void* y, int64_t B,
                                              int64_t T, int64_t C, int64_t H,
                                              int64_t W, int64_t R, int residual,
                                              dsc_dtype_t dtype,
                                              uint64_t wait_limit_ns, void* stream);
dsc_status_t dsc_lowrank_bwd_selftest_timeout(
    const void* x, const void* z, const void* U, const void* dy, void* dx,
    void* dz, void* dU, void* workspace, size_t workspace_bytes, int64_t B,
    int64_t T, int64_t C, int64_t H, int64_t W, int64_t R, int residual,
    dsc_dtype_t dtype, uint64_t wait_limit_ns, void* stream);

/*
 * Self-test of the failure path of the tcgen05 kernel behind
 * dsc_headwise_proj_decode (bf16 batches of 17 or more sequences; its CTAs
 * form clusters that meet at cluster barriers).  As above: every bounded
 * wait limited to wait_limit_ns (1 us .. 1 s) and a producer that issues no
 * loads, so the MMA issuer's wait runs out; every CTA still reaches both
 * cluster barriers, frees its TMEM and returns.  Expected result: DSC_OK,
 * then dsc_device_error reports 2 (or 3), y and state are unspecified, and
 * the next normal call runs correctly.  Arguments as for
 * dsc_headwise_proj_decode plus wait_limit_ns; DSC_ERR_UNSUPPORTED when the
 * call would not take the tcgen05 kernel (fp32, or fewer than 17
 * sequences), DSC_ERR_INVALID_ARG for B = 0 or a limit outside the range.
 */
dsc_status_t dsc_headwise_proj_decode_selftest_timeout(
    const void* h, const void* Wp, const void* w, void* state, void* y, int64_t B, int64_t D,
    int64_t C, int64_t H, int64_t W, int residual, dsc_dtype_t dtype, uint64_t wait_limit_ns,
    void* stream);

/*
 * Largest workspace dsc_lowrank_bwd_noalloc can provide: 32 MiB.
 */
#define DSC_LOWRANK_BWD_NOALLOC_MAX_BYTES ((size_t)32 << 20)

/*
 * dsc_lowrank_bwd for callers that cannot allocate device memory.  The
 * paper has no counterpart to this entry point; it exists for library
 * users.  Some callers cannot call cudaMalloc: a plugin inside a host
 * program that owns all device memory, a service with a fixed memory budget
 * that forbids allocation after start-up, or a latency-critical path that
 * cannot afford the device synchronisation an allocation may cause.  This
 * variant takes no workspace argument; it uses a fixed 32 MiB array compiled
 * into the library (every GPU that loads the library holds it until the
 * process exits) and calls no allocating routine.
 *   Arguments, layouts, results and errors are those of dsc_lowrank_bwd.
 *   A problem whose workspace (dsc_lowrank_bwd_workspace_size) exceeds
 *   DSC_LOWRANK_BWD_NOALLOC_MAX_BYTES is refused with DSC_ERR_WORKSPACE
 *   before anything is enqueued; use dsc_lowrank_bwd for it.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any
 *   stream capture.  The stream must belong to the current device.  The
 *   address is kept for the life of the process: after cudaDeviceReset (or
 *   anything else that destroys and recreates the device's primary context)
 *   this entry point must not be called again on that device.
 *   All calls share the one array: two calls whose work overlaps on the GPU
 *   (different streams, or different host threads, without ordering between
 *   them) race on it and give wrong results.  Calls ordered on one stream
 *   are safe; nothing needs clearing between them, since every partial sum
 *   is written before it is read.
 */
dsc_status_t dsc_lowrank_bwd_noalloc(const void* x, const void* z,
                                     const void* U, const void* dy, void* dx,
                                     void* dz, void* dU, int64_t B, int64_t T,
                                     int64_t C, int64_t H, int64_t W,
                                     int64_t R, int residual,
                                     dsc_dtype_t dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSC_H_ */
