/*
 * libsa -- Stochastic Attention (SA) forward pass on NVIDIA GB300 (sm_103a).
 *
 * What the library computes ("Stochastic Attention" technical summaries,
 * gist.science/ja/paper/2604.00754 and gist.science/ko/paper/2604.00754):
 *
 *   SA   ("Core mechanism", steps 1-3): permute the rows of Q, K and V by a
 *        random permutation sigma, X'[p] = X[sigma[p]]; run sliding-window
 *        attention over the permuted rows with the window |p - q| <= h,
 *        h = floor(w / 2), truncated at the sequence ends; scatter the result
 *        back, Y[sigma[p]] = Y'[p].  The causal variant ("Theoretical
 *        properties", causal-constraint bullet) additionally keeps only keys
 *        with sigma[q] <= sigma[p], i.e. keys that precede the query in the
 *        ORIGINAL order (the query itself included).
 *   SWA  ("Problem statement"): token i attends to keys [max(0, i-w+1), i].
 *   Gated dual path ("Gated SA and SWA", the displayed equation):
 *        Y = sigmoid(a_sa) * Y_sa + sigmoid(a_swa) * Y_swa, with the gate
 *        logits a_sa, a_swa given per token and query head.
 *
 * Softmax weights are exp(scale * <q, k>) normalised over the window;
 * scale defaults to 1/sqrt(head_dim).  Grouped-query attention: query head
 * hq uses kv head hq / (num_q_heads / num_kv_heads).
 *
 * Layouts (all row-major and contiguous, "BSHD"):
 *   q    bf16  [batch, seqlen, num_q_heads,  head_dim]
 *   k, v bf16  [batch, seqlen, num_kv_heads, head_dim]
 *   out  bf16  [batch, seqlen, num_q_heads,  head_dim]
 *   perm int32 [batch, seqlen]   sigma of each sequence (shared by all heads)
 *   gate logits fp32 [batch, seqlen, num_q_heads], indexed by ORIGINAL token.
 *
 * Ownership and execution: the caller owns every buffer.  Device pointers
 * must come from the CUDA device that is current on the calling thread.  The
 * forward calls enqueue kernels on `stream` and return without waiting; they
 * allocate no memory.  The library keeps a thread-local detail string for the
 * last error (sa_last_error_message) and one device-side error word of its
 * own that is used when a call is given a NULL error word.
 *
 * Errors: argument checks run on the host before anything is launched and
 * return SA_ERR_INVALID_ARG or SA_ERR_UNSUPPORTED.  A failed launch returns
 * SA_ERR_CUDA.  Faults detected on the device (a perm entry outside [0, n),
 * a duplicate perm entry, a pipeline wait that ran past its limit) are OR-ed
 * into a device error word as SA_ERRBIT_* bits; sa_check_error() reads it.
 * No call traps, aborts or waits without a bound.
 */
#ifndef LIBSA_H
#define LIBSA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sa_status {
  SA_OK = 0,
  SA_ERR_INVALID_ARG = 1, /* NULL pointer, size <= 0, Hq % Hkv != 0, ... */
  SA_ERR_UNSUPPORTED = 2, /* valid request this library cannot run (head_dim, alignment, kernel) */
  SA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  SA_ERR_BAD_PERM = 4,    /* device check found perm entries out of range or repeated */
  SA_ERR_TIMEOUT = 5,     /* a device pipeline wait ran past its bound; results are invalid */
  SA_ERR_INTERNAL = 6     /* a device self-check of an internal index failed (a library bug) */
} sa_status_t;

/* Kernel choice (sa_params_t.kernel). */
enum {
  SA_KERNEL_AUTO = 0,    /* a tcgen05 tensor-core kernel when the shape fits one, else SIMT */
  SA_KERNEL_SIMT = 1,    /* CUDA-core kernel: any window, the correctness baseline */
  SA_KERNEL_TCGEN05 = 2, /* the better-fitting tcgen05 kernel; SA_ERR_UNSUPPORTED if none fits */
  SA_KERNEL_TCGEN05_GATHER = 3, /* tcgen05 kernel that gathers every window with TMA */
  SA_KERNEL_TCGEN05_RING = 4,   /* tcgen05 kernel with a sliding K/V ring (spans <= 256 keys
                                   whose rings fit shared memory) */
  SA_KERNEL_TCGEN05_CHUNK = 5   /* tcgen05 kernel streaming the span in 128-key chunks with an
                                   online softmax (any window) */
};

/* Bits of the device error word. */
#define SA_ERRBIT_RANGE 1   /* a perm entry outside [0, seqlen) */
#define SA_ERRBIT_DUP 2     /* two positions of perm name the same token */
#define SA_ERRBIT_TIMEOUT 4 /* a bounded pipeline wait gave up */
#define SA_ERRBIT_INTERNAL 8 /* an internal index self-check failed (a library bug); access skipped */

typedef struct sa_params {
  int32_t batch;        /* B >= 1 */
  int32_t seqlen;       /* n >= 1 */
  int32_t num_q_heads;  /* Hq >= 1, a multiple of num_kv_heads */
  int32_t num_kv_heads; /* Hkv >= 1 */
  int32_t head_dim;     /* d: 64 or 128 */
  int32_t window;       /* w >= 1.  SA: half-width h = w / 2 (floor).  SWA: w keys. */
  int32_t window_swa;   /* gated call only: SWA window; <= 0 means "same as window" */
  int32_t causal;       /* SA: 0 = window only, 1 = also sigma[q] <= sigma[p] */
  float softmax_scale;  /* <= 0 means 1/sqrt(head_dim) */
  int32_t kernel;       /* SA_KERNEL_* */
  int32_t* err;         /* device int32 error word, or NULL for the library's own */
} sa_params_t;

/*
 * Stochastic Attention forward ("Core mechanism" steps 1-3; causal rule from
 * "Theoretical properties").  Reads q, k, v (bf16, BSHD), perm (device int32
 * [B, n], must be a permutation of [0, n) per sequence; the forward kernels
 * trust it, validate it first with sa_inverse_perm + sa_check_error if it is
 * untrusted), writes every row of out (bf16 [B, n, Hq, d]).  out must not
 * alias q, k or v.  All device pointers 16-byte aligned.
 */
sa_status_t sa_forward(const sa_params_t* params, const void* q, const void* k, const void* v,
                       const int32_t* perm, void* out, cudaStream_t stream);

/*
 * Sliding-window attention over the original order ("Problem statement"):
 * token i attends to keys [max(0, i - window + 1), i].  Same layouts and
 * rules as sa_forward; params->causal is ignored (SWA is always causal).
 */
sa_status_t swa_forward(const sa_params_t* params, const void* q, const void* k, const void* v,
                        void* out, cudaStream_t stream);

/*
 * Gated SA + SWA dual path ("Gated SA and SWA" equation):
 *   out = sigmoid(gate_sa_logits) * SA(q,k,v; perm, window, causal)
 *       + sigmoid(gate_swa_logits) * SWA(q,k,v; window_swa)
 * Gate logits: device fp32 [B, n, Hq], indexed by original token and query
 * head, broadcast over head_dim.  The merge happens in place in out (the SWA
 * term is written first, the SA term is added by the second kernel), so the
 * workspace is unused: pass NULL / 0 (sa_gated_workspace_size returns 0).
 * Rounding: on the tensor-core kernels the SWA term is stored in out as bf16
 * and the SA pass adds its term in fp32 and rounds again (two bf16
 * roundings); the CUDA-core kernel (SA_KERNEL_SIMT) merges in registers and
 * rounds once.
 */
sa_status_t sa_swa_gated_forward(const sa_params_t* params, const void* q, const void* k,
                                 const void* v, const int32_t* perm, const float* gate_sa_logits,
                                 const float* gate_swa_logits, void* out, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

/* Bytes of device workspace sa_swa_gated_forward needs for these params (0). */
size_t sa_gated_workspace_size(const sa_params_t* params);

/*
 * Backward pass.  The summary pretrains a model from scratch with the gated
 * SA + SWA pair ("Main contributions", item 3; "Results", first bullet),
 * which needs the gradients of each path's output; they follow from the
 * forward definitions above by the chain rule.  Given the upstream gradient
 * dout (bf16 [B, n, Hq, d], the gradient of the loss with respect to out),
 * a call writes
 *   dq bf16 [B, n, Hq, d],  dk, dv bf16 [B, n, Hkv, d]
 * (the kv-head gradients summed over the query heads that read them) and,
 * for the gated call, the gate-logit gradients dgate_* fp32 [B, n, Hq]
 * (NULL skips one).  Softmax normalisers are recomputed from q and k; the
 * forward outputs are not needed.  Every row of dq, dk, dv is written.
 * Layouts and pointer rules as for the forward calls; outputs must not alias
 * inputs or each other.  Caller-owned device workspace of at least the
 * *_workspace_size bytes, 256-byte aligned, contents ignored on entry.
 * Supported: head_dim 64 or 128, Hq/Hkv dividing 128, and a key span of at
 * most 256 per 128-row tile (128/g + 2*floor(w/2) keys for SA, 128/g + w - 1
 * for SWA); else SA_ERR_UNSUPPORTED.  params->kernel must be SA_KERNEL_AUTO
 * or SA_KERNEL_TCGEN05.  Asynchronous on `stream` (2 kernel launches per
 * path; 7 for the gated call).
 */
sa_status_t sa_backward(const sa_params_t* params, const void* q, const void* k, const void* v,
                        const int32_t* perm, const void* dout, void* dq, void* dk, void* dv,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);
sa_status_t swa_backward(const sa_params_t* params, const void* q, const void* k, const void* v,
                         const void* dout, void* dq, void* dk, void* dv, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream);
/* Workspace of sa_backward / swa_backward: two fp32 values per (token, query head). */
size_t sa_backward_workspace_size(const sa_params_t* params);

/*
 * sa_backward without a workspace argument and without any allocation.  The
 * pages have no counterpart to this call: it exists for callers that cannot
 * allocate device memory at the point where they run the backward pass --
 * for example a training or serving loop whose device memory is reserved
 * once at start-up, a host framework that owns every device allocation and
 * hands the library only tensors, or a plain C caller with no allocator of
 * its own.  The scratch that sa_backward takes from its workspace (two fp32
 * values per (token, query head)) lives instead in a fixed device array
 * inside this library, sized for batch * seqlen * num_q_heads <= 1048576
 * (8 MiB, held on every device that loads the library until the process
 * exits).  Larger problems return SA_ERR_UNSUPPORTED with a message naming
 * the limit; use sa_backward for them.  Arguments, results and the other
 * rules are those of sa_backward; the call itself allocates nothing.  The
 * first call on each device looks up the array's address on that device, so
 * make that first call before any stream capture.  Every call on a device
 * shares the one array: calls whose kernels may overlap on the GPU (different
 * streams without ordering between them) race on it, so order them.  The
 * array keeps the last call's contents; each call writes every value it
 * reads first, so nothing is cleared between calls.
 */
sa_status_t sa_backward_noalloc(const sa_params_t* params, const void* q, const void* k,
                                const void* v, const int32_t* perm, const void* dout, void* dq,
                                void* dk, void* dv, cudaStream_t stream);

/*
 * Gradients of the gated dual path ("Gated SA and SWA" equation).  The
 * gate-logit gradient of a row is g (1 - g) <dout, Y_path> with g its
 * sigmoid.  The two paths' dq, dk, dv are summed in fp32 in the workspace and
 * rounded to bf16 once.
 */
sa_status_t sa_swa_gated_backward(const sa_params_t* params, const void* q, const void* k,
                                  const void* v, const int32_t* perm,
                                  const float* gate_sa_logits, const float* gate_swa_logits,
                                  const void* dout, void* dq, void* dk, void* dv, float* dgate_sa,
                                  float* dgate_swa, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream);
/* Workspace of sa_swa_gated_backward: the above plus fp32 dq, dk and dv. */
size_t sa_swa_gated_backward_workspace_size(const sa_params_t* params);

/*
 * sigma^{-1} ("Core mechanism" step 3; "Theoretical properties": an O(n)
 * index operation): inv[b, perm[b, p]] = p for every sequence b.  perm and
 * inv are device int32 [batch, n] and must not overlap.  Entries of perm
 * outside [0, n) set SA_ERRBIT_RANGE, repeated entries set SA_ERRBIT_DUP in
 * *d_err (device int32; NULL selects the library's own word); inv is then
 * unspecified.  Asynchronous on `stream`; read the verdict with
 * sa_check_error.
 */
sa_status_t sa_inverse_perm(const int32_t* perm, int32_t* inv, int32_t batch, int32_t n,
                            int32_t* d_err, cudaStream_t stream);

/*
 * The gate logits of the dual path ("Gated SA and SWA": the two paths are
 * mixed through independent sigmoid projections).  Both projections of the
 * layer input x (bf16 [tokens, d_model], row-major; tokens = B * n in BSHD
 * token order) in one tensor-core GEMM:
 *   gate_sa_logits  = x W_sa^T  + b_sa,   gate_swa_logits = x W_swa^T + b_swa,
 * W_* bf16 [num_q_heads, d_model], b_* fp32 [num_q_heads] or NULL, outputs
 * fp32 [tokens, num_q_heads] -- exactly the logits sa_swa_gated_forward and
 * sa_swa_gated_backward take (they apply the sigmoid).  d_model a multiple
 * of 64, num_q_heads <= 128, x and weights 16-byte aligned.  fp32
 * accumulation of bf16 products.  Asynchronous on `stream`.
 */
sa_status_t sa_gate_projection(const void* x, int32_t tokens, int32_t d_model,
                               int32_t num_q_heads, const void* w_sa, const void* w_swa,
                               const float* b_sa, const float* b_swa, float* gate_sa_logits,
                               float* gate_swa_logits, int32_t* d_err, cudaStream_t stream);

/*
 * Rotary position embedding by ORIGINAL token index, applied in place to a
 * bf16 BSHD tensor (Q or K) before the sigma-gather, so that a score depends
 * on the distance i - j between the two tokens in the original order
 * whatever permutation brings them into one window.  Convention: for
 * k < head_dim/2 the pair (x_k, x_{k + head_dim/2}) of token i is rotated by
 * the angle i * base^(-2k/head_dim).  head_dim even and <= 128, base > 1.
 * Angles are reduced in fp64, rotations done in fp32, results rounded to
 * bf16.  Any 2-byte-aligned x is accepted (16-byte aligned data takes the
 * widest accesses).  Asynchronous on `stream`.
 */
sa_status_t sa_rope(void* x, int32_t batch, int32_t seqlen, int32_t heads, int32_t head_dim,
                    double base, cudaStream_t stream);

/*
 * Receptive fields of L stacked SA layers ("Theoretical properties",
 * receptive-field bullet: with an independent sigma per layer the field grows
 * far faster than sliding-window attention's and covers the sequence in
 * O(log_w n) layers).  With N_l(i) the neighbour set of token i in layer l
 * (window `window`, causal or not, as in sa_forward) and R_0(i) = {i},
 * R_l(i) = union over j in N_l(i) of R_{l-1}(j); layer 1 acts first on the
 * inputs, so R_L(i) applies layer L to {i}, then L-1, ..., 1.
 *   perms    device int32 [layers, n]: sigma of each layer (one sequence)
 *   targets  device int32 [num_targets]: tokens whose fields are measured
 *   sizes    device int64 [layers, num_targets] out: sizes[l-1][t] = |R_l(targets[t])|
 * Exact integer counts.  Workspace: sa_receptive_field_workspace_size(n)
 * bytes, 16-byte aligned.  1 <= layers <= 64, floor(window/2) <= 1024.  Perm
 * or target entries outside [0, n) set SA_ERRBIT_RANGE in *d_err (NULL: the
 * library's word).  Asynchronous on `stream`.
 */
size_t sa_receptive_field_workspace_size(int32_t n);
sa_status_t sa_receptive_field(const int32_t* perms, int32_t layers, int32_t n, int32_t window,
                               int32_t causal, const int32_t* targets, int32_t num_targets,
                               int64_t* sizes, void* workspace, size_t workspace_bytes,
                               int32_t* d_err, cudaStream_t stream);

/*
 * Host routing plan of sigma-routed sequence sharding: one sequence split
 * over `world` ranks (one per GPU) with chunk c = ceil(n / world).  Rank r
 * holds the original tokens [r c, (r+1) c) of Q, K, V and of the output, and
 * computes the SA rows of the permuted positions [r c, (r+1) c) ("Core
 * mechanism": sliding-window attention over the permuted order), working on
 * the span [r c - floor(w/2), (r+1) c + floor(w/2)) clipped to [0, n).
 *   tokens      out [span]: the span's tokens in ascending original order --
 *               the local rows of Q, K and V that rank r gathers from their
 *               owners (token t lives on rank t / c)
 *   local_perm  out [span]: local row of the token at span position j; the
 *               relabelling is monotone, so sa_forward on (local rows,
 *               local_perm, the same window and causal rule) computes the
 *               owned positions' rows exactly as the whole sequence would
 *   span_begin  out: first permuted position of the span
 *   own_begin, own_end  out: the permuted positions rank r owns; their rows
 *               are local rows local_perm[own - span_begin] of the local
 *               output, for tokens perm[own], returned to their owners
 * capacity >= sa_shard_span(n, window, world, rank).  perm_host is the
 * whole sigma (host int32 [n]) and must be a permutation (SA_ERR_BAD_PERM
 * otherwise).  Host only, O(n + span log span).
 */
int32_t sa_shard_span(int32_t n, int32_t window, int32_t world, int32_t rank);
sa_status_t sa_shard_plan(const int32_t* perm_host, int32_t n, int32_t window, int32_t world,
                          int32_t rank, int32_t* tokens, int32_t* local_perm, int32_t capacity,
                          int32_t* span_begin, int32_t* own_begin, int32_t* own_end);

/*
 * Host: draw sigma ~ Uniform(S_n) for (seed, layer, batch_index) ("Core
 * mechanism" step 1: one independent permutation per layer) into perm_host
 * (int32[n], caller-owned).  Generator: the stream state is the output of one
 * splitmix64 step applied to seed + (layer << 32) + batch_index; then a
 * Durstenfeld Fisher-Yates shuffle of the identity, i = n-1 .. 1, swapping
 * positions i and j = (x * (i + 1)) >> 64 for each splitmix64 output x.
 * layer and batch_index must be >= 0.  Runs on the calling thread; no GPU.
 */
sa_status_t sa_make_perm(uint64_t seed, int32_t layer, int32_t batch_index, int32_t n,
                         int32_t* perm_host);

/*
 * Synchronise `stream`, read the device error word (NULL: the library's own)
 * and map it to a status: SA_ERR_INTERNAL if SA_ERRBIT_INTERNAL is set, else
 * SA_ERR_TIMEOUT if SA_ERRBIT_TIMEOUT is set, else SA_ERR_BAD_PERM if a perm
 * bit is set, else SA_OK.  The word is left as is.
 */
sa_status_t sa_check_error(const int32_t* d_err, cudaStream_t stream);

/* Enqueue a reset of the device error word (NULL: the library's own) to 0. */
sa_status_t sa_clear_error(int32_t* d_err, cudaStream_t stream);

/*
 * Failure detection: every pipeline wait inside the tcgen05 kernels is
 * bounded by a number of SM cycles; a wait that runs past it sets
 * SA_ERRBIT_TIMEOUT in the device error word, the kernel stops its pipeline,
 * lets its own copies and MMAs finish, frees its tensor memory and returns
 * (sa_check_error then reports SA_ERR_TIMEOUT; the CUDA context stays usable).
 * sa_set_wait_limit sets that bound for every launch made from now on, by any
 * thread; cycles <= 0 restores the default (4e9 cycles, ~2 s at the maximum
 * SM clock).  A bound far below a kernel's normal waits (a few hundred cycles)
 * makes a call give up on purpose, which is how the timeout path is tested.
 * The final wait for a kernel's own MMAs before tensor memory is freed has a
 * fixed bound of its own and is not affected.  Host only; never fails.
 */
sa_status_t sa_set_wait_limit(int64_t cycles);

/* The current wait bound in SM cycles (see sa_set_wait_limit). */
int64_t sa_get_wait_limit(void);

/* Static text for a status code. */
const char* sa_status_string(sa_status_t status);

/* Detail of the last failing call on this thread ("" if none). */
const char* sa_last_error_message(void);

/* SA_KERNEL_SIMT, SA_KERNEL_TCGEN05_GATHER, SA_KERNEL_TCGEN05_RING or
 * SA_KERNEL_TCGEN05_CHUNK: the kernel the last successful forward call on
 * this thread launched (0 before any; for the gated path, the SA pass's). */
int32_t sa_last_kernel(void);

/* Number of kernel launches the last successful forward or backward call on
 * this thread made (forward: 1 for SA/SWA, 2 for the gated path; backward:
 * 2 per path, 7 for the gated call). */
int32_t sa_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBSA_H */
