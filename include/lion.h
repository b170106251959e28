/*
 * lion.h -- C ABI of liblion.so, the GB300 (sm_103a) implementation of the
 * LION bidirectional masked linear-attention operator.
 *
 * The operator (rebuttal page "LION: A bidirectional framework that trains
 * like a Transformer and infers like an RNN", reply "Concern 1",
 * Theorem 3.3 Eq 25):
 *
 *     Y = SCALE( (phi(Q) phi(K)^T) (.) M ) V
 *
 * per (batch b, head h), rows i, j in [0, L):
 *   s_ij = phi(q_i) . phi(k_j)
 *   M_ij = prod_{t = min(i,j)+1}^{max(i,j)} lambda_t,   M_ii = 1
 *   y_i  = sum_j M_ij s_ij v_j / sum_j M_ij s_ij          (SCALE = row sum)
 *
 * Masks (rebuttal page, list of running examples; "LION Part IV - Results"):
 *   LION_MASK_LIT  lambda = 1, M all ones ("LION-LIT" / "LION-fire").
 *   LION_MASK_D    one fixed lambda per head, M_ij = lambda_h^|i-j|
 *                  ("LION-D" / "LION-RETNET").
 *   LION_MASK_S    a lambda per token ("LION-S", selective).
 * Feature maps (rebuttal page, reply "4) Default non-linearity"):
 *   elu(x)+1 for LIT and D, SiLU followed by an L2 normalisation over the
 *   head dimension (norm clamped below at 1e-12) for S.
 * Forms, all computing the same Y (Theorem 3.3; blog "LION Chunk"):
 *   LION_FORM_FULL   quadratic attention with the mask generated on the fly.
 *   LION_FORM_RNN    forward and backward recurrences (Theorem 3.3 Eq 20-24)
 *                    keeping only y^{F/B}_i and c^{F/B}_i (reply "1:
 *                    Recurrence Form", O(Ld + L) memory).
 *   LION_FORM_CHUNK  chunkwise: masked attention inside chunks of `chunk`
 *                    tokens, chunk states carried by forward and backward
 *                    scans.
 *
 * Conventions shared by every entry point
 *   - Tensors are row-major and contiguous.  q, k, v, out: [B][H][L][d].
 *   - log_lambda holds log(lambda) (finite, <= 0): LIT ignores it (NULL
 *     allowed); D: [H]; S: [B][H][L].  All float32.
 *   - out is float32 (bfloat16 when lion_args.out_bf16 asks for it).  Every
 *     pointer is memory owned by the caller: device memory, except the
 *     host buffers that lion_attn_fwd_host takes.
 *   - Calls are asynchronous on `stream`.  Argument errors are detected on
 *     the host before anything is launched and return a status; nothing is
 *     written then.  A launch or runtime failure returns LION_ERR_CUDA.
 *   - d must be 16, 32, 64 or 128.  q, k, v, out and workspace must be
 *     16-byte aligned.
 *   - The library keeps no state between calls except a per-device cache of
 *     device properties and of resolved driver entry points, the device
 *     status word that lion_sync_status reads and clears, and the fixed
 *     scratch array of lion_attn_fwd_rnn_noalloc.
 */
#ifndef LION_H_
#define LION_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LION_OK = 0,
  LION_ERR_INVALID_ARG = 1,  /* null pointer, bad enum, size or alignment   */
  LION_ERR_UNSUPPORTED = 2,  /* valid request this build does not handle   */
  LION_ERR_CUDA = 3,         /* a CUDA call or kernel launch failed        */
  LION_ERR_NO_MEMORY = 4,    /* workspace allocation failed                */
  LION_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up         */
  LION_ERR_RANGE = 6         /* a value exceeded the fp16 range (65504) of a
                                tensor-core operand: v, or (seen through a
                                non-finite row sum) unbounded features or a
                                masked score; the output of that call is not
                                valid                                        */
} lion_status;

typedef enum { LION_MASK_LIT = 0, LION_MASK_D = 1, LION_MASK_S = 2 } lion_mask_kind;
typedef enum { LION_FORM_FULL = 0, LION_FORM_RNN = 1, LION_FORM_CHUNK = 2 } lion_form;
typedef enum { LION_DTYPE_BF16 = 0, LION_DTYPE_FP32 = 1 } lion_dtype;
typedef enum {
  LION_PHI_DEFAULT = 0,   /* elu+1 for LIT and D, SiLU + L2 for S */
  LION_PHI_ELU1 = 1,
  LION_PHI_SILU_L2 = 2,
  LION_PHI_IDENTITY = 3   /* phi(x) = x */
} lion_phi;

/* Largest L the FULL form accepts (its cost is O(L^2 d)); larger L returns
 * LION_ERR_UNSUPPORTED. */
#define LION_FULL_MAX_L 8192

/*
 * lion_attn_fwd -- the operator for bfloat16 q, k, v.
 *   q, k, v     [B][H][L][d] bfloat16, device.
 *   log_lambda  see conventions (device; NULL for LIT).
 *   mask_kind   lion_mask_kind.   form: lion_form.
 *   chunk       chunk length for LION_FORM_CHUNK, 1 <= chunk <= 1024 (larger:
 *               LION_ERR_UNSUPPORTED).  The result does not depend on it up
 *               to rounding.  With d = 64, chunk 64 and chunk 128 run on the
 *               tensor cores at any L (chunk 128: one launch for L <= 256,
 *               three above); every other chunk, and d != 64, runs on the
 *               CUDA cores in fp32.  Ignored by the other forms.
 *   out         [B][H][L][d] float32, device, written entirely.
 * Workspace, when the form needs one, is taken from the stream-ordered
 * allocator (cudaMallocAsync/cudaFreeAsync on `stream`); use
 * lion_attn_fwd_ex to pass one instead.
 */
lion_status lion_attn_fwd(const void* q, const void* k, const void* v,
                          const float* log_lambda, int B, int H, int L, int d,
                          int mask_kind, int form, int chunk, float* out,
                          cudaStream_t stream);

/* Every option of the operator in one struct. */
typedef struct {
  const void* q;             /* [B][H][L][d], dtype below                  */
  const void* k;
  const void* v;
  const float* log_lambda;   /* see conventions                            */
  float* out;                /* [B][H][L][d] float32                       */
  int B, H, L, d;
  int mask_kind;             /* lion_mask_kind                             */
  int form;                  /* lion_form                                  */
  int chunk;                 /* LION_FORM_CHUNK only                       */
  int dtype;                 /* lion_dtype of q, k, v                      */
  int phi;                   /* lion_phi                                   */
  void* workspace;           /* device, 256-byte aligned, or NULL          */
  size_t workspace_bytes;    /* >= lion_attn_workspace_bytes(...) if given */
  cudaStream_t stream;
  int out_bf16;              /* 0: out is float32; 1: out is bfloat16      */
} lion_args;

/*
 * lion_attn_fwd_ex -- as lion_attn_fwd with a dtype (BF16 or FP32 inputs), a
 * feature-map override, an optional caller workspace and an optional
 * bfloat16 output.  With workspace == NULL the library allocates what it
 * needs stream-ordered.
 *   out_bf16 = 1: out is [B][H][L][d] bfloat16 (16-byte aligned), each value
 *   the fp32 result rounded to nearest even (the arithmetic is unchanged).
 *   The chunk-128 tensor-core kernels (bf16 inputs, d = 64, chunk = 128)
 *   store it themselves, which halves their output bytes; every other path
 *   computes into a stream-ordered fp32 temporary of B*H*L*d floats
 *   (allocated by the library, not part of the workspace) and rounds it.
 *   lion_attn_fwd_causal takes the field the same way.
 */
lion_status lion_attn_fwd_ex(const lion_args* a);

/* Workspace bytes lion_attn_fwd_ex needs for this problem (0 if none). */
size_t lion_attn_workspace_bytes(int B, int H, int L, int d, int form, int chunk);

/*
 * lion_attn_fwd_causal -- the forward half alone, for a unidirectional
 * (generative) model: y_i = sum_{j<=i} M_ij s_ij v_j / sum_{j<=i} M_ij s_ij.
 * This is the causal Linear-Transformer recurrence with the decay (rebuttal
 * page reply "1: Recurrence Form"; the unidirectional LION-S of reply
 * "Q5").  Arguments as lion_attn_fwd_ex, in every form (FULL: keys up to the
 * row; RNN: the forward recurrence alone; CHUNK: the forward chunk scan and
 * the lower triangle of each chunk).  Computed on the CUDA cores in fp32,
 * chunk <= 1024.  Workspace: lion_attn_workspace_bytes of the form (B*H*L
 * floats for RNN and CHUNK, plus the features of every token for RNN (whose
 * size also holds the bidirectional form's backward sums, unused here), for
 * CHUNK with chunk <= 64, and for FULL at d = 64 and 128, which needs
 * nothing else; NULL: stream-ordered allocation).
 */
lion_status lion_attn_fwd_causal(const lion_args* a);

/*
 * lion_rnn_step -- one token of one direction of the recurrent form, for
 * B*H heads at once (Theorem 3.3 Eq 20-24; the causal Linear-Transformer
 * recurrence of reply "1: Recurrence Form" with a decay):
 *     S <- lambda * S + phi(k) v^T,    z <- lambda * z + phi(k)
 *     y_part = phi(q)^T S,             c_part = phi(q)^T z
 *   q, k, v     [B][H][d] in `dtype` (lion_dtype), device.
 *   log_lambda  LIT: ignored; D: [H]; S: [B][H] (this token's lambda; for
 *               the backward direction pass lambda of the token after it).
 *   S           [B][H][d][d] float32, row m = feature of phi(k), updated in place;
 *               16-byte aligned (LION_ERR_INVALID_ARG otherwise).
 *   z           [B][H][d] float32, updated in place.
 *   y_part      [B][H][d] float32 out;  c_part [B][H] float32 out.
 * The caller owns the state.  Combining the two directions into y_i uses
 * y_i = (yF_i + yB_i - s_ii v_i) / (cF_i + cB_i - s_ii), s_ii = phi(q_i).phi(k_i).
 */
lion_status lion_rnn_step(const void* q, const void* k, const void* v,
                          const float* log_lambda, float* S, float* z,
                          float* y_part, float* c_part, int B, int H, int d,
                          int mask_kind, int dtype, cudaStream_t stream);

/*
 * lion_sync_status -- synchronise `stream`, then report whether any kernel
 * of this library on the current device gave up on a bounded device-side
 * wait since the last call (LION_ERR_TIMEOUT), was given a traversal order
 * that is not a permutation (LION_ERR_INVALID_ARG), or, on the tensor-core
 * chunk path, met a value its fp16 operands cannot hold (LION_ERR_RANGE: use
 * LION_DTYPE_FP32, or a chunk length the CUDA cores take); the flag is then
 * cleared.
 * Kernels never spin unboundedly: a wait that runs out records the error,
 * releases its tensor memory and returns.  LION_ERR_CUDA if the
 * synchronisation itself fails.
 */
lion_status lion_sync_status(cudaStream_t stream);

/*
 * lion_attn_fwd_rnn_noalloc -- the recurrent form (LION_FORM_RNN, default
 * feature map) for callers that cannot allocate device memory: code inside
 * a host framework that owns all device memory through its own allocator,
 * or a latency-critical loop that must not call cudaMalloc/cudaFree (which
 * may synchronise the device).  The paper has no counterpart; this is an
 * interface convenience of this library.
 *   Arguments as lion_attn_fwd_ex with form = LION_FORM_RNN; dtype is
 *   LION_DTYPE_BF16 or LION_DTYPE_FP32 for q, k, v.
 *   Scratch: a fixed device array of this library holding one float per
 *   head-token, so B * H * L <= LION_NOALLOC_MAX_HEAD_TOKENS (4 MiB array,
 *   held on every GPU that loads the library until the process exits);
 *   larger problems return LION_ERR_UNSUPPORTED before anything launches.
 *   Nothing is allocated, ever.  The first call on a device looks up the
 *   array's device address (cudaGetSymbolAddress) for that device: make it
 *   before any stream capture.  The address is kept for the life of the
 *   process, so a cudaDeviceReset after the first call is not supported.
 *   Every call shares the array; calls that overlap on the GPU (unordered
 *   streams) race on it -- order them.  Argument checks and errors are those
 *   of lion_attn_fwd_ex.
 */
#define LION_NOALLOC_MAX_HEAD_TOKENS (1u << 20)
lion_status lion_attn_fwd_rnn_noalloc(const void* q, const void* k, const void* v,
                                      const float* log_lambda, int B, int H, int L, int d,
                                      int mask_kind, int dtype, float* out,
                                      cudaStream_t stream);

/*
 * lion_attn_bwd -- gradients of a scalar loss through the operator, given
 * dy = dLoss/dY (the training path: the full form trains like a Transformer,
 * rebuttal page reply "Concern 1", Theorem 3.3 Eq 25).  With A = (phi(Q)
 * phi(K)^T) (.) M, num = A V, den = A 1 and Y = num / den row by row:
 *     dnum_i = dy_i / den_i,   dden_i = -(dy_i . y_i) / den_i,
 *     dA_ij = dnum_i . v_j + dden_i,   dV = A^T dnum,
 *     dphi(Q) = (M (.) dA) phi(K),     dphi(K) = (M (.) dA)^T phi(Q),
 *     dlog(lambda_u) = sum of A_ij dA_ij over the pairs (i, j) with
 *                      min(i,j) < u <= max(i,j)   (the factors of M_ij),
 * then through the feature map by the chain rule.  The result does not
 * depend on which form produced Y (they agree, Theorem 3.3).
 *   q, k, v      [B][H][L][d] in `dtype`, device; log_lambda as for the forward.
 *   dy           [B][H][L][d] float32, device.
 *   dq, dk, dv   [B][H][L][d] float32, device, written entirely.
 *   dlog_lambda  LIT: unused (NULL allowed); D: [H] (summed over the batch
 *                and the positions, which share lambda_h); S: [B][H][L]
 *                (position 0 never enters the mask: 0).  float32, device.
 * Computed in fp32 on the CUDA cores, O(L^2 d) per head like the full form
 * (L <= LION_FULL_MAX_L, else LION_ERR_UNSUPPORTED).  Workspace: as
 * lion_attn_fwd_ex (NULL: stream-ordered allocation).
 */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  const float* log_lambda;
  const float* dy;
  float* dq;
  float* dk;
  float* dv;
  float* dlog_lambda;
  int B, H, L, d;
  int mask_kind;             /* lion_mask_kind                             */
  int dtype;                 /* lion_dtype of q, k, v                      */
  int phi;                   /* lion_phi                                   */
  void* workspace;           /* device, 256-byte aligned, or NULL          */
  size_t workspace_bytes;    /* >= lion_attn_bwd_workspace_bytes(...)      */
  cudaStream_t stream;
} lion_bwd_args;
lion_status lion_attn_bwd(const lion_bwd_args* a);

/* Workspace bytes lion_attn_bwd needs for this problem. */
size_t lion_attn_bwd_workspace_bytes(int B, int H, int L, int d);

/*
 * lion_attn_bwd_chunk -- the same gradients as lion_attn_bwd through the
 * chunkwise form, for any L (the forms agree, Theorem 3.3; "LION Part IV -
 * Results", "LION Chunk").  Each gradient is a product of the masked
 * structure the forward scans: inside chunks of 64 tokens (32 at d = 128) the
 * masked score and dA tiles, across chunks the forward and backward states of
 * phi(k) [v; 1]^T and of phi(q) G^T (G_i = [dy_i / den_i ; -(dy_i . y_i) /
 * den_i]), each a d x (d + 1) fp32 matrix per chunk, carried by scans as in
 * Theorem 3.3 Eq 20-24.  dlog_lambda from the row and column terms as in
 * lion_attn_bwd.
 *   Arguments, layouts and errors as lion_attn_bwd, without its length limit.
 *   Computed in fp32 on the CUDA cores, O(L d^2 + L C d) per head.  Workspace
 *   as returned by lion_attn_bwd_chunk_workspace_bytes (about 2 (d + 4)^2 / C
 *   + d + 7 floats per head-token; NULL: stream-ordered allocation).
 */
lion_status lion_attn_bwd_chunk(const lion_bwd_args* a);

/* Workspace bytes lion_attn_bwd_chunk needs for this problem (0 if invalid). */
size_t lion_attn_bwd_chunk_workspace_bytes(int B, int H, int L, int d);

/*
 * lion_attn_fwd_host -- lion_attn_fwd_ex on inputs and output in host memory.
 * The library cuts the batch into `slices` slices (0: min(B, 4)) and, with two
 * device buffer sets, copies slice s in on one internal stream, runs the
 * operator on it on `stream` and copies its output out on another, so that
 * copies in, compute and copies out of neighbouring slices overlap.  Every
 * copy is a single cudaMemcpyAsync of a contiguous slice.
 *   q, k, v, log_lambda, out: host memory with the layouts of lion_args.
 *   Page-locked memory (cudaHostAlloc / cudaHostRegister) is needed for the
 *   overlap; pageable memory is accepted and copied synchronously.  Device
 *   memory is refused (LION_ERR_INVALID_ARG): use lion_attn_fwd_ex.
 *   Other fields as lion_args.  Device memory for the slices is allocated
 *   stream-ordered on `stream` and freed in its order.
 * Asynchronous like the other entry points: work already queued on `stream`
 * comes first, later work on `stream` comes after the last copy out, and out
 * is complete once `stream` is synchronised.  The host buffers must stay
 * valid until then.
 */
typedef struct {
  const void* q;             /* host [B][H][L][d], dtype below             */
  const void* k;
  const void* v;
  const float* log_lambda;   /* host, as lion_args                         */
  float* out;                /* host [B][H][L][d] float32                  */
  int B, H, L, d;
  int mask_kind;             /* lion_mask_kind                             */
  int form;                  /* lion_form                                  */
  int chunk;                 /* LION_FORM_CHUNK only                       */
  int dtype;                 /* lion_dtype of q, k, v                      */
  int phi;                   /* lion_phi                                   */
  int slices;                /* batch slices (0: the library picks)        */
  cudaStream_t stream;
} lion_host_args;
lion_status lion_attn_fwd_host(const lion_host_args* a);

/*
 * lion_attn_fwd_reordered -- the full form with the mask averaged over two
 * traversal orders of the tokens: LION-S (v2) and the reordered-patch LION-D
 * and LION-S (rebuttal page reply "P2: Comparison against vision SSMs",
 * item 1: the masks of two traversals of the patch grid are averaged; results
 * page "LION Part IV - Results", "Model Comparisons").
 *   Along order p, position t holds token order[p*L + t]; the mask between
 *   two tokens is the operator's mask of the sequence taken in that order
 *   (the product of the decays at the positions after the earlier token, up
 *   to and including the later one; LION-D: lambda to the distance between
 *   the positions).  y_i = sum_j M_ij s_ij v_j / sum_j M_ij s_ij with
 *   M = (M^1 + M^2) / 2.  Identical orders give the plain operator run on the
 *   reordered sequence; LIT ignores the orders.
 *   q, k, v, log_lambda, out, B, H, L, dtype, phi, workspace, stream: as
 *   lion_args (form and chunk are not used).
 *   order   device int32 [2][L], each row a permutation of 0..L-1, the same
 *           for every (b, h); 4-byte aligned.  A row that is not a
 *           permutation is detected on the device: the call still returns
 *           LION_OK, every access stays in bounds, out is undefined, and the
 *           next lion_sync_status returns LION_ERR_INVALID_ARG.
 *   Computed in fp32 on the CUDA cores; d in {64, 128} (else
 *   LION_ERR_UNSUPPORTED) and L <= LION_FULL_MAX_L.  Workspace as returned
 *   by lion_attn_reordered_workspace_bytes (NULL: stream-ordered allocation).
 */
typedef struct {
  const void* q;             /* [B][H][L][d], dtype below                  */
  const void* k;
  const void* v;
  const float* log_lambda;   /* as lion_args                               */
  const int* order;          /* [2][L] device int32                        */
  float* out;                /* [B][H][L][d] float32                       */
  int B, H, L, d;
  int mask_kind;             /* lion_mask_kind                             */
  int dtype;                 /* lion_dtype of q, k, v                      */
  int phi;                   /* lion_phi                                   */
  void* workspace;           /* device, 256-byte aligned, or NULL          */
  size_t workspace_bytes;
  cudaStream_t stream;
} lion_reorder_args;
lion_status lion_attn_fwd_reordered(const lion_reorder_args* a);

/* Workspace bytes lion_attn_fwd_reordered needs (0 if d is not 64 or 128). */
size_t lion_attn_reordered_workspace_bytes(int B, int H, int L, int d);

/*
 * lion_attn_bwd_reordered -- gradients of a scalar loss through
 * lion_attn_fwd_reordered, given dy = dLoss/dy: the same products as
 * lion_attn_bwd with the averaged mask, and for the decays the derivative
 * of each order's mask (the product of the decays that order passes)
 * taken along that order.
 *   q, k, v, log_lambda, order, B, H, L, d, mask_kind, dtype, phi: as
 *   lion_reorder_args; dy, dq, dk, dv, dlog_lambda: as lion_bwd_args.
 *   A row of order that is not a permutation is reported as for the forward
 *   (every access stays in bounds, the next lion_sync_status returns
 *   LION_ERR_INVALID_ARG).  fp32 on the CUDA cores; d in {64, 128} (else
 *   LION_ERR_UNSUPPORTED), L <= LION_FULL_MAX_L.  Workspace as returned by
 *   lion_attn_reordered_bwd_workspace_bytes (NULL: stream-ordered allocation).
 */
typedef struct {
  const void* q;             /* [B][H][L][d], dtype below                  */
  const void* k;
  const void* v;
  const float* log_lambda;   /* as lion_args                               */
  const int* order;          /* [2][L] device int32                        */
  const float* dy;           /* [B][H][L][d] float32                       */
  float* dq;                 /* [B][H][L][d] float32                       */
  float* dk;
  float* dv;
  float* dlog_lambda;        /* as lion_bwd_args                           */
  int B, H, L, d;
  int mask_kind;             /* lion_mask_kind                             */
  int dtype;                 /* lion_dtype of q, k, v                      */
  int phi;                   /* lion_phi                                   */
  void* workspace;           /* device, 256-byte aligned, or NULL          */
  size_t workspace_bytes;
  cudaStream_t stream;
} lion_reorder_bwd_args;
lion_status lion_attn_bwd_reordered(const lion_reorder_bwd_args* a);

/* Workspace bytes lion_attn_bwd_reordered needs (0 if d is not 64 or 128). */
size_t lion_attn_reordered_bwd_workspace_bytes(int B, int H, int L, int d);

/*
 * Testing aids for the bound on device-side waits (no counterpart in the
 * pages; not needed in normal use).
 * lion_debug_set_wait_cycles -- the bound, in SM clock cycles, on every
 *   mbarrier wait of the tensor-core kernels launched after the call
 *   (process-wide).  0 restores the default of 2e9 cycles (about 1 s);
 *   negative values return LION_ERR_INVALID_ARG.  A bound far below a
 *   kernel's normal waits makes it give up and report LION_ERR_TIMEOUT.
 * lion_debug_wait_timeout -- launches one warp on `stream` that waits, with
 *   that bound, on an mbarrier that nothing arrives at, through the same
 *   wait the kernels use.  No copy and no matrix product is in flight in it:
 *   the wait gives up, the kernel records the timeout and returns, and the
 *   next lion_sync_status returns LION_ERR_TIMEOUT (clearing the flag).
 *   With the default bound the call lasts about a second.
 */
lion_status lion_debug_set_wait_cycles(long long cycles);
lion_status lion_debug_wait_timeout(cudaStream_t stream);

/* Static, human-readable text for a status. */
const char* lion_status_string(lion_status s);

/* Version of this ABI (bumped on any incompatible change). */
int lion_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LION_H_ */
