/*
 * bsa.h -- C ABI of libbsa.so: GB300 (sm_103a) fused causal attention forwards.
 *
 * Two forwards, each one CUDA kernel launch that never materialises the T x T
 * score matrix:
 *
 *   tra_forward         threshold rectified attention (TRA)
 *   nsa_select_forward  NSA selection-branch attention
 *
 * plus the TRA backward, the differential TRA, the NSA selection forward
 * in the page's block-outer split-K form (nsa_select_forward_fsa, which works
 * in a caller-provided workspace) and tra_forward_host, which takes host
 * buffers and streams them through the GPU.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is caller-owned DEVICE memory (cudaMalloc or a
 *   framework allocator) on the current device, except the host tensors of
 *   tra_forward_host.  Tensors are dense, contiguous
 *   and row-major in the shapes given below; there are no stride arguments.
 *   q, k, v and out start on a 16-byte boundary.
 * - The library never synchronises: work is enqueued on `stream` (0 = legacy
 *   default stream) and the call returns after the launch.  It allocates no
 *   device memory, except tra_diff_forward with normalize != 0, which takes a
 *   small temporary through the stream-ordered allocator (documented there).
 *   Its state is a device error word per kernel file, written only when a
 *   bounded wait times out (see bsa_device_error), and the streams and
 *   events tra_forward_host creates on its first call on a device.  Inputs must stay valid and
 *   unmodified, and outputs untouched by others, until that work completes.
 * - A call returns a bsa_status.  Argument errors are detected on the host
 *   before anything is enqueued and leave every buffer untouched.  A launch
 *   failure returns BSA_ERR_LAUNCH.  Nothing aborts or prints.
 * - Out-of-range values inside the index tensor (see nsa_select_forward) are
 *   a precondition violation: the kernel treats any negative index as padding
 *   and never reads outside k/v for an index >= T / block_size (such a slot is
 *   skipped), but results for such a row are unspecified.
 */
#ifndef BSA_H
#define BSA_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define BSA_API __attribute__((visibility("default")))
#else
#define BSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of q, k, v and out. */
typedef enum {
  BSA_F32 = 0,  /* IEEE float32 */
  BSA_BF16 = 1  /* bfloat16 (8-bit exponent, 7-bit mantissa) */
} bsa_dtype;

typedef enum {
  BSA_OK = 0,
  BSA_ERR_NULLPTR = 1,     /* a required pointer is NULL                     */
  BSA_ERR_SHAPE = 2,       /* a size is out of range or inconsistent          */
  BSA_ERR_DTYPE = 3,       /* dtype is not a bsa_dtype                        */
  BSA_ERR_UNSUPPORTED = 4, /* a valid request this build does not implement,
                              or a parameter outside the method (p <= 0,
                              non-finite beta)                               */
  BSA_ERR_LAUNCH = 5,      /* the CUDA launch failed (cudaGetLastError)       */
  BSA_ERR_DEVICE = 6,      /* no usable sm_100-family device / driver entry   */
  BSA_ERR_ALIGN = 7,       /* a tensor pointer is not 16-byte aligned         */
  BSA_ERR_MEMORY = 8,      /* a temporary scratch buffer could not be
                              allocated or released (tra_diff_forward)       */
  BSA_ERR_SCRATCH_LIMIT = 9 /* the problem needs more scratch than the fixed
                              buffer of tra_diff_forward_noalloc holds        */
} bsa_status;

/*
 * tra_forward -- threshold rectified attention forward.
 *
 * Defined on the page "triton_threshold_attention.py" (snap-research/TDA):
 * module docstring formula and the forward kernel _threshold_rela_fwd_kernel.
 * For every (b, h) and query row i = 0..T-1:
 *
 *   tau(i)      = beta * sqrt(2 * ln(i + 1) / D)        (computed in fp32)
 *   out[b,h,i,:] = sum_{j <= i} ReLU(q_i . k_j - tau(i))^p * v_j
 *
 * Causal, unnormalised, no 1/sqrt(D) factor on q.k.  p == 1 and p == 2 use
 * the identity and a product; any other p > 0 uses x^p = exp2(p * log2 x).
 * A masked (future) pair contributes nothing for every beta (the page's own
 * code agrees for beta >= 0).
 *
 *   q, k, v, out : [B, H, T, D], element type `dtype`; out has the input type
 *                  (the page casts its fp32 result back to the input dtype).
 *   B, H, T      : >= 1; B * H <= 2^31 - 1 and B*H*T*D < 2^40.
 *   D            : a multiple of 16 from 16 to 128 (head dim; the page's
 *                  kernel takes the head dim as its BLOCK_D).  Head dims
 *                  below 64 run the width-64 bf16 kernel and 80 .. 112 the
 *                  width-128 one, on zero-filled columns.
 *   beta         : finite.      p : finite and > 0.
 *   dtype        : BSA_BF16 -- tensor-core (tcgen05) path, bf16 operands,
 *                  fp32 accumulation, weights rounded to bf16 before W.V;
 *                  BSA_F32  -- fp32 CUDA-core path (fp32 FMA throughout).
 *   stream       : CUDA stream the kernel is enqueued on.
 *
 * Errors: BSA_ERR_NULLPTR, BSA_ERR_SHAPE (sizes), BSA_ERR_DTYPE,
 * BSA_ERR_UNSUPPORTED (D not a multiple of 16 in 16..128, p <= 0,
 * non-finite beta/p),
 * BSA_ERR_ALIGN, BSA_ERR_DEVICE, BSA_ERR_LAUNCH.
 */
BSA_API int tra_forward(const void* q, const void* k, const void* v, void* out,
                        int B, int H, int T, int D, float beta, float p,
                        int dtype, cudaStream_t stream);

/* Flags of tra_forward_ex. */
typedef enum {
  /* p = k + 1/2 with k in 0..3 (0.5, 1.5, 2.5, 3.5) is evaluated as
     x^k * sqrt(x): one square root per score instead of exp2(p * log2 x). */
  BSA_TRA_SQRT_HALF_POWERS = 1
} bsa_tra_flags;

/*
 * tra_forward_ex -- tra_forward with evaluation flags.
 *
 * Same method, arguments, layout, rules and errors as tra_forward, plus
 * `flags`, a bitwise OR of bsa_tra_flags (0 = exactly tra_forward; unknown
 * bits return BSA_ERR_UNSUPPORTED).  With BSA_TRA_SQRT_HALF_POWERS and
 * dtype BSA_BF16, a half-integer p from 0.5 to 3.5 runs x^k * sqrt(x) on the
 * pair kernel; the result is the same map ReLU(.)^p within rounding (the
 * square root is correct to about one float ulp).  Other p, and dtype
 * BSA_F32, are computed exactly as tra_forward computes them.  The page
 * evaluates every non-integer power through exp and log, which tra_forward
 * follows; this option is an equivalent evaluation for half-integer powers.
 */
BSA_API int tra_forward_ex(const void* q, const void* k, const void* v,
                           void* out, int B, int H, int T, int D, float beta,
                           float p, int dtype, int flags, cudaStream_t stream);

/*
 * tra_forward_host -- tra_forward on tensors in host memory.
 *
 * Same method, arguments, layout, rules and errors as tra_forward, except
 * that q, k, v (read) and out (written) are HOST pointers.  The (b, h) heads
 * are streamed through the GPU in about eight chunks: the host-to-device
 * copies of one chunk, the kernel of the previous chunk and the
 * device-to-host copy of the one before overlap on three library streams
 * (created on the first call on a device and kept for the process).  For the
 * copies to overlap, the host buffers should be page-locked (cudaHostAlloc
 * or cudaHostRegister); pageable buffers give the same result with the
 * copies serialised.  The call is asynchronous with respect to `stream`:
 * work already queued on `stream` comes first, and out is complete when
 * `stream` reaches the point after the call (synchronize `stream` before
 * reading out or reusing q, k, v, out or the workspace).
 *
 *   workspace, workspace_bytes : caller-owned device memory, 256-byte
 *       aligned, at least tra_forward_host_workspace_size(B, H, T, D, dtype)
 *       bytes (three stages of q, k, v and out for one chunk of heads).
 *
 * Errors: those of tra_forward, plus BSA_ERR_NULLPTR for a NULL workspace,
 * BSA_ERR_ALIGN for a misaligned workspace and BSA_ERR_SCRATCH_LIMIT for a
 * workspace that is too small.  Host pointers need no particular alignment.
 */
BSA_API size_t tra_forward_host_workspace_size(int B, int H, int T, int D,
                                               int dtype);
BSA_API int tra_forward_host(const void* q, const void* k, const void* v,
                             void* out, int B, int H, int T, int D,
                             float beta, float p, int dtype, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/*
 * tra_backward -- gradients of the threshold rectified attention forward.
 *
 * Defined on the page "triton_threshold_attention.py": ThresholdRelaFunction
 * .backward with the kernels _threshold_rela_bwd_kernel_dq and
 * _threshold_rela_bwd_kernel_dkv.  With x_ij = q_i . k_j - tau(i) over the
 * causal pairs j <= i and dout the gradient of out:
 *
 *   W_ij  = ReLU(x_ij)^p                    dv_j = sum_i W_ij dout_i
 *   dA_ij = (dout_i . v_j) p ReLU(x_ij)^(p-1)   (0 where x_ij <= 0)
 *   dq_i  = sum_j dA_ij k_j                 dk_j = sum_i dA_ij q_i
 *
 * beta and p receive no gradient (as on the page).  Scores are recomputed
 * (nothing is saved by tra_forward).
 *
 * bf16: one fused kernel computes the scores and dout . v of every (key tile,
 * query tile) pair once; dk and dv accumulate on chip, and each pair's dq
 * partial is added (fp32) into a temporary of 4 * B * H * T * D bytes, taken
 * with cudaMallocFromPoolAsync on `stream` from the library's memory pool
 * (as tra_diff_forward's) and returned with cudaFreeAsync on `stream`; a
 * zeroing kernel before and a conversion kernel after it run on `stream` too.  The
 * order of the fp32 dq additions varies between runs, so dq may differ in
 * its last bf16 bit from one run to the next; dk and dv do not.  For results
 * that repeat bit for bit use tra_backward_ex with
 * BSA_TRA_BWD_DETERMINISTIC.  fp32: two launches (CUDA-core kernels, fp32
 * throughout, as the page computes; deterministic).
 *
 *   q, k, v, dout       : [B, H, T, D] inputs of `dtype` (dout = dL/d out).
 *   dq, dk, dv          : [B, H, T, D] outputs of `dtype` (fp32 accumulation);
 *                         they must not alias the inputs or each other.
 *   D                   : as for tra_forward (a multiple of 16 up to 128;
 *                         below the tile width on zero-filled columns).
 *   B, H, T, beta, p    : as for tra_forward.  For 0 < p < 1 the derivative
 *                         p x^(p-1) grows without bound as x -> 0+, so a
 *                         score within rounding of tau(i) makes dq and dk
 *                         ill-conditioned (any two correct evaluations may
 *                         differ there).
 *   dtype               : BSA_BF16 or BSA_F32.
 *
 * Errors: as for tra_forward (BSA_ERR_UNSUPPORTED for other D),
 * plus BSA_ERR_MEMORY if the bf16 temporary cannot be allocated or released.
 */
BSA_API int tra_backward(const void* q, const void* k, const void* v,
                         const void* dout, void* dq, void* dk, void* dv,
                         int B, int H, int T, int D, float beta, float p,
                         int dtype, cudaStream_t stream);

/* Flags of tra_backward_ex. */
typedef enum {
  /* bf16: the two-kernel form (one block per key tile for dk and dv, one per
     query tile for dq, each producing the scores itself).  It allocates
     nothing and repeats bit for bit; it does 14 D instead of 10 D tensor
     FLOPs per causal pair. */
  BSA_TRA_BWD_DETERMINISTIC = 1
} bsa_tra_bwd_flags;

/*
 * tra_backward_ex -- tra_backward with evaluation flags.
 *
 * Same method, arguments, layout, rules and errors as tra_backward, plus
 * `flags`, a bitwise OR of bsa_tra_bwd_flags (0 = exactly tra_backward;
 * unknown bits return BSA_ERR_UNSUPPORTED).  BSA_TRA_BWD_DETERMINISTIC
 * allocates nothing, so it never returns BSA_ERR_MEMORY.  fp32 ignores the
 * flag (its kernels are deterministic and allocate nothing).
 */
BSA_API int tra_backward_ex(const void* q, const void* k, const void* v,
                            const void* dout, void* dq, void* dk, void* dv,
                            int B, int H, int T, int D, float beta, float p,
                            int dtype, int flags, cudaStream_t stream);

/*
 * tra_diff_forward -- threshold differential attention forward.
 *
 * Defined on the page "triton_threshold_attention.py":
 * differential_threshold_rela_triton.  With n(x) = x / max(||x||_2, 1e-12)
 * applied row by row when `normalize` is non-zero (identity otherwise):
 *
 *   out = TRA(n(q1), n(k1), v) - clamp(lambda, 0, 1) * TRA(n(q2), n(k2), v)
 *
 * where TRA is tra_forward's map with the same beta and p.  One fused kernel
 * runs both score streams on the same query tile and shares each V tile;
 * each stream accumulates its P.V product in fp32 and the two are combined
 * (first minus clamp(lambda, 0, 1) times second) before the bf16 store.
 * With normalize (bf16), a pre-pass kernel first writes bf16 copies of k1
 * and k2 with their rows normalised (as the page normalises q and k before
 * its kernel), into a temporary of 4 * B * H * T * D bytes; the kernel reads
 * those copies and scales each score by 1/max(||q_i||, 1e-12), which it
 * computes from its own query tile.  The temporary is
 * taken with cudaMallocFromPoolAsync on `stream` and returned with
 * cudaFreeAsync on `stream`, from a memory pool the library creates on the
 * device at first use (it keeps up to 1 GiB of freed temporaries mapped; the
 * caller's default pool is not touched); without
 * normalize nothing is allocated.  BSA_F32 runs one CUDA-core kernel that
 * folds the two row norms into each score (q.k times both reciprocals) and
 * allocates nothing in either mode.
 *
 *   q1, q2, k1, k2, v, out : [B, H, T, D] of `dtype` (out may not alias
 *                            inputs).
 *   D                      : as for tra_forward.
 *   B, H, T, beta, p       : as for tra_forward.
 *   lambda                 : any non-NaN value; clamped to [0, 1].
 *   dtype                  : BSA_BF16 or BSA_F32.
 *
 * Errors: as for tra_forward, plus BSA_ERR_MEMORY if the temporary cannot be
 * allocated or released.
 */
BSA_API int tra_diff_forward(const void* q1, const void* q2, const void* k1,
                             const void* k2, const void* v, void* out,
                             int B, int H, int T, int D, float beta,
                             float lambda, float p, int normalize, int dtype,
                             cudaStream_t stream);

/*
 * tra_diff_backward -- gradients of tra_diff_forward (page
 * "triton_threshold_attention.py", differential_threshold_rela_triton,
 * differentiated through its normalisation, its two ThresholdRelaFunction
 * calls and the clamp of lambda).  With a = n(q), b = n(k) (row-wise L2
 * normalisation x / max(||x||, 1e-12) when normalize, else the identity) and
 * c = clamp(lambda, 0, 1):
 *   out = TRA(a1, b1, v) - c TRA(a2, b2, v),
 *   dv  = dv1 - c dv2, (da1, db1, dv1) = tra_backward(a1, b1, v, dout),
 *   (da2, db2, dv2) = -c ... of tra_backward(a2, b2, v, dout) (TRA's gradients
 *   are linear in dout), dq1 = n'(q1)^T da1 etc. through the normalisation,
 *   dlambda = -sum(dout * TRA(a2, b2, v)) for 0 < lambda < 1, else 0,
 *   summed as -sum(v * W2^T dout), W2^T dout being the dv of
 *   tra_backward(a2, b2, v, dout) before the -c (the same sum regrouped,
 *   TRA(a2, b2, v) = W2 v), so it needs no forward pass.
 * bf16 runs the fused tcgen05 backward twice on normalised bf16 copies of
 * q1, q2, k1, k2 (taken from the inputs in fp32 and rounded once) and takes
 * the gradients through the normalisation in fp32; BSA_F32 the CUDA-core
 * kernels.  Temporaries (the copies and both passes' gradients, their dq in
 * fp32: for bf16 the fused backward's accumulators, read without a
 * conversion) come from the library's stream-ordered pool as for
 * tra_diff_forward.  The dq outputs, like tra_backward's, may differ in
 * their last bf16 bit between runs (fp32 partials added in a run-dependent
 * order); so may dlambda (one atomic addition per block).
 *
 *   q1, q2, k1, k2, v, dout        : [B, H, T, D] of `dtype` (inputs).
 *   dq1, dq2, dk1, dk2, dv         : [B, H, T, D] of `dtype` (outputs; they
 *                                    must not alias the inputs or each other).
 *   dlambda                        : device float (4-byte aligned) written
 *                                    with dlambda, or NULL to skip it.
 *   B, H, T, D, beta, lambda, p,
 *   normalize, dtype               : as for tra_diff_forward.
 *
 * Errors: as for tra_diff_forward (BSA_ERR_NULLPTR for any null tensor,
 * BSA_ERR_ALIGN for a tensor not 16-byte aligned or a misaligned dlambda),
 * plus BSA_ERR_MEMORY.
 */
BSA_API int tra_diff_backward(const void* q1, const void* q2, const void* k1,
                              const void* k2, const void* v,
                              const void* dout, void* dq1, void* dq2,
                              void* dk1, void* dk2, void* dv, float* dlambda,
                              int B, int H, int T, int D, float beta,
                              float lambda, float p, int normalize, int dtype,
                              cudaStream_t stream);

/*
 * tra_diff_forward_noalloc -- tra_diff_forward without any allocation.
 *
 * The source pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate device memory from inside the call: code whose
 * device memory is owned by its own allocator (a framework that reserves the
 * GPU up front and accounts for every byte), or code on a latency-critical
 * path that must not wait on the CUDA allocator.  It computes the same map
 * as tra_diff_forward, with the same arguments, rules and errors, but the
 * row normalisation factors go to a fixed scratch array that the library
 * holds in device memory (16 MiB on every GPU that loads the library, until
 * the process exits) instead of a temporary from a memory pool, and there is
 * no room there for normalised copies of k1 and k2: with normalize the
 * kernel scales each score by the key row's factor as well as the query
 * row's, in fp32, instead of reading keys normalised and rounded to bf16.
 * So with normalize the two entry points agree within bf16 rounding, not
 * bit for bit (each is bit-repeatable on its own); without normalize they
 * run the same kernel and agree exactly.  It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *
 * Limit: with normalize != 0 the problem must satisfy
 *   B * H * Tp <= 1,048,576   (Tp = T rounded up to a multiple of 128);
 * larger problems return BSA_ERR_SCRATCH_LIMIT before anything is enqueued.
 * Without normalize no scratch is used and there is no such limit.
 *
 * Set-up: the first call on a device looks up the device address of the
 * array (cudaGetSymbolAddress, with that device current) and caches it; make
 * that first call before any stream capture on that device.
 *
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents.  Each call rewrites every entry it reads before reading it,
 * so nothing needs clearing, but calls whose work overlaps on the GPU (for
 * example on two streams at once) race on the array and give undefined
 * results: serialise them.
 */
BSA_API int tra_diff_forward_noalloc(const void* q1, const void* q2,
                                     const void* k1, const void* k2,
                                     const void* v, void* out, int B, int H,
                                     int T, int D, float beta, float lambda,
                                     float p, int normalize, int dtype,
                                     cudaStream_t stream);

/*
 * nsa_select_forward -- NSA selection-branch attention forward (bf16).
 *
 * Defined on the page "nsa_selection_kernel.py" (openbox-llm): module
 * docstring "The operation", the ground truth selection_forward_reference and
 * the log-sum-exp of _selection_fwd_kernel.  With G = Hq / Hkv and query head
 * h reading kv head h / G, for every (b, h, i):
 *
 *   J     = { j : j / block_size is a non-negative entry of
 *                 block_idx[b, h/G, i, 0..S-1], and j <= i }
 *   s_j   = (q[b,h,i] . k[b,h/G,j]) * D^-0.5
 *   out[b,h,i] = sum_{j in J} softmax(s)_j * v[b,h/G,j]     (0 if J is empty)
 *   lse[b,h,i] = ln sum_{j in J} exp(s_j)                   (-1e9 if J empty)
 *
 *   q, out     : [B, Hq, T, D] bf16.      k, v : [B, Hkv, T, D] bf16.
 *   block_idx  : [B, Hkv, T, S] int32, shared by the G heads of a group;
 *                -1 = padding.  A row is read as a set, as the page's
 *                reference does: a block listed more than once is selected
 *                once, and the order of the slots does not matter.
 *   lse        : [B, Hq, T] fp32, or NULL to skip it.
 *   D          : 16, 32, 64 or 128 (the page: a power of two <= 128).
 *   block_size : 16, 32, 64 or 128 (the page: >= 16; its tiles need a power
 *                of two).  64-token blocks of 64 or 128 dims run a TMA kernel,
 *                every other shape a cp.async one; results agree either way.
 *   1 <= S <= 32.
 *   T          : multiple of block_size.   Hq % Hkv == 0, 1 <= Hq / Hkv <= 16.
 *   stream     : CUDA stream the kernel is enqueued on.
 *
 * Errors: BSA_ERR_NULLPTR (q, k, v, block_idx or out NULL), BSA_ERR_SHAPE,
 * BSA_ERR_UNSUPPORTED (other D, block_size or group size), BSA_ERR_ALIGN,
 * BSA_ERR_DEVICE, BSA_ERR_LAUNCH.
 */
BSA_API int nsa_select_forward(const void* q, const void* k, const void* v,
                               const int32_t* block_idx, void* out, float* lse,
                               int B, int Hq, int Hkv, int T, int D,
                               int block_size, int S, cudaStream_t stream);

/*
 * nsa_select_forward_fsa -- the same NSA selection forward in the block-outer
 * split-K form (bf16).
 *
 * Defined on the page "nsa_selection_kernel.py" (openbox-llm), FSA forward
 * section (_selection_fwd_blockouter_kernel, selection_forward_fsa).  Every
 * selected key block's K/V is read once: for each (query i, live block j of
 * its row) pair and head h of the group, a softmax partial over the block's
 * tokens t <= i,
 *
 *   m = max_t s_t,   l = sum_t exp(s_t - m),   acc = sum_t exp(s_t - m) v_t,
 *
 * (s_t as in nsa_select_forward) is written to the workspace, and a
 * log-sum-exp combine per (b, h, i) gives
 *
 *   out = sum_j w_j acc_j / sum_j w_j l_j,   w_j = exp(m_j - max_j m_j),
 *   lse = max_j m_j + ln sum_j w_j l_j,
 *
 * which is the same softmax over the union of the selected causal tokens as
 * nsa_select_forward computes (out = 0, lse = -1e9 for a row with no pair).
 * A live slot holds 0 <= j < T / block_size with j * block_size <= i, and
 * is the first slot of its row that holds j (set semantics: a repeated block
 * forms one pair).
 *
 * Arguments, shapes, dtypes, preconditions and errors are those of
 * nsa_select_forward (but only block_size 64 with D 64 or
 * 128 is built: other shapes return BSA_ERR_UNSUPPORTED), plus:
 *   workspace       : caller-owned device memory of at least
 *                     nsa_select_fsa_workspace_size(...) bytes, 256-byte
 *                     aligned; overwritten, and in use until the work on
 *                     `stream` completes (one workspace per concurrent call).
 *   workspace_bytes : its size.
 * Extra errors: BSA_ERR_NULLPTR (workspace NULL), BSA_ERR_ALIGN (workspace
 * not 256-byte aligned), BSA_ERR_SCRATCH_LIMIT (workspace_bytes too small),
 * BSA_ERR_SHAPE (B * Hq * T * S >= 2^31).
 *
 * nsa_select_fsa_workspace_size returns the bytes of workspace needed for
 * these sizes, or 0 if nsa_select_forward_fsa does not accept them; it is
 * host only and touches no device.
 *
 * The work is six kernel launches on `stream`: the inverted selection lists
 * are built on the device (count, scan, fill), then the block-outer pass and
 * the combine.  The workspace holds B * Hq * T * S * (D + 2) floats of
 * partials plus the lists (about 4.4 GB at B=2, Hq=32, T=8192, S=16, D=128).
 */
BSA_API size_t nsa_select_fsa_workspace_size(int B, int Hq, int Hkv, int T,
                                             int D, int block_size, int S);
BSA_API int nsa_select_forward_fsa(const void* q, const void* k,
                                   const void* v, const int32_t* block_idx,
                                   void* out, float* lse, int B, int Hq,
                                   int Hkv, int T, int D, int block_size,
                                   int S, void* workspace,
                                   size_t workspace_bytes,
                                   cudaStream_t stream);

/* Static, NUL-terminated description of a bsa_status value (never NULL). */
BSA_API const char* bsa_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
BSA_API int bsa_version(void);

/*
 * bsa_device_error -- read and clear the library's device-side error words.
 *
 * Every wait inside the kernels (on a TMA arrival, an MMA completion or a
 * sibling warp) is bounded to about one second; a wait that runs out records
 * code 1 here and the kernel winds down instead of hanging (its outputs are
 * then unspecified); a kernel that finds its shared memory misaligned records
 * code 2 and does nothing.  Returns 0 when no kernel has failed since the
 * last call, else the largest code recorded, -1 if the words could not be
 * read.  Synchronises
 * with the current device (cudaMemcpyFromSymbol); not for the hot path.
 */
BSA_API int bsa_device_error(void);

/*
 * Self tests: device code paths the attention calls reach only in rare
 * conditions, run on their own so that a test can check them on the GPU.
 * The pages have no counterpart of these; they serve this library's tests.
 *
 * bsa_selftest_wait_timeout -- one thread of a one-CTA kernel waits, with a
 * limit of `limit_cycles` SM clocks (1 .. 1e8), on an mbarrier that nothing
 * arrives on, through the same bounded wait every kernel uses.  The wait
 * gives up, records code 1 in the library's device error word (read it with
 * bsa_device_error) and writes 0 to *result (1 would mean the wait completed,
 * which cannot happen); the kernel then returns.  No copy or tensor-core
 * operation is in flight, so the context stays usable.  `result` is a device
 * int (4-byte aligned).  Errors: BSA_ERR_NULLPTR, BSA_ERR_SHAPE (limit out of
 * range), BSA_ERR_ALIGN, BSA_ERR_DEVICE, BSA_ERR_LAUNCH.
 *
 * bsa_selftest_log2 -- for n floats x (device memory), writes the
 * general-power epilogue's FMA-pipe log2 (exponent/mantissa split and a
 * degree-5 minimax polynomial, the path POW_GENERAL_MIX uses for part of the
 * scores) to y_fma and CUDA's log2f to y_ref.  Inputs are meant to be
 * non-negative finite floats.  Errors: BSA_ERR_NULLPTR, BSA_ERR_SHAPE (n < 1),
 * BSA_ERR_ALIGN (a pointer not 4-byte aligned), BSA_ERR_DEVICE,
 * BSA_ERR_LAUNCH.
 *
 * bsa_selftest_exp2 -- for n floats y (device memory), writes the
 * general-power epilogue's FMA-pipe exp2 (y clamped to [-127, 128], rounding
 * to an integer n and a degree-4 minimax polynomial for 2^(y - n), the path
 * POW_GENERAL_MIX uses for part of the scores) to w_fma, in fp32 before the
 * epilogue's bf16 rounding, and CUDA's exp2f to w_ref.  y = -127 (and below)
 * gives +0.0 exactly, y = 128 (and above) +inf.  Errors as for
 * bsa_selftest_log2.
 */
BSA_API int bsa_selftest_wait_timeout(long long limit_cycles, int* result,
                                      cudaStream_t stream);
BSA_API int bsa_selftest_log2(const float* x, float* y_fma, float* y_ref,
                              int n, cudaStream_t stream);
BSA_API int bsa_selftest_exp2(const float* y, float* w_fma, float* w_ref,
                              int n, cudaStream_t stream);

/*
 * bsa_read_probe -- a measurement helper, not part of the method (the pages
 * have no counterpart): reads `bytes` (a multiple of 16, at most 2^40) of
 * device memory at `buf` (16-byte aligned) `reps` times (1 .. 100000) with
 * 16-byte loads that bypass L1, over a grid of four CTAs per SM, and XORs
 * what it read into the device word *sink (4-byte aligned).  Timed with CUDA
 * events on `stream`, bytes * reps / time is the read bandwidth of wherever
 * the buffer lives: for a buffer that fits in L2 and was read once before,
 * the L2 read bandwidth that the NSA selection gathers are served from.
 * Errors: BSA_ERR_NULLPTR, BSA_ERR_SHAPE, BSA_ERR_ALIGN, BSA_ERR_DEVICE,
 * BSA_ERR_LAUNCH.
 */
BSA_API int bsa_read_probe(const void* buf, size_t bytes, int reps,
                           unsigned int* sink, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BSA_H */
