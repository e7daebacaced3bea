// C-ABI entry points of libsa: argument validation, kernel choice, the host
// sigma generator (sigma ~ Uniform(S_n), one per layer: Stochastic Attention
// summary, "Core mechanism" step 1) and error reporting.  Every step of the
// attention itself runs in the CUDA kernels of sa_tc_ring.cu, sa_tc_chunk.cu,
// sa_tc.cu and sa_simt.cu; sigma^-1 in sa_perm.cu.
#include <atomic>
#include <mutex>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "sa_internal.h"

namespace sa {

static thread_local char g_msg[512] = "";
static thread_local int32_t g_last_kernel = 0;
static thread_local int32_t g_last_launches = 0;

__device__ int32_t g_error_word = 0;

constexpr long long kDefaultWaitLimit = 4000000000LL;  // ~2 s at the maximum SM clock
static std::atomic<long long> g_wait_limit{kDefaultWaitLimit};

long long wait_limit_cycles() { return g_wait_limit.load(std::memory_order_relaxed); }

sa_status_t fail(sa_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

int32_t* default_error_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
  return static_cast<int32_t*>(p);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared shape checks of the three forward calls.
static sa_status_t check_params(const sa_params_t* prm, bool need_window) {
  if (prm == nullptr) return fail(SA_ERR_INVALID_ARG, "params is NULL");
  if (prm->batch < 1 || prm->seqlen < 1 || prm->num_q_heads < 1 || prm->num_kv_heads < 1)
    return fail(SA_ERR_INVALID_ARG, "batch, seqlen and head counts must be >= 1");
  if (prm->num_q_heads % prm->num_kv_heads != 0)
    return fail(SA_ERR_INVALID_ARG, "num_q_heads (%d) must be a multiple of num_kv_heads (%d)",
                prm->num_q_heads, prm->num_kv_heads);
  if (prm->head_dim != 64 && prm->head_dim != 128)
    return fail(SA_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", prm->head_dim);
  if (need_window && prm->window < 1) return fail(SA_ERR_INVALID_ARG, "window must be >= 1");
  if (prm->kernel < SA_KERNEL_AUTO || prm->kernel > SA_KERNEL_TCGEN05_CHUNK)
    return fail(SA_ERR_INVALID_ARG, "unknown kernel selector %d", prm->kernel);
  const double rows = double(prm->batch) * prm->seqlen * prm->num_q_heads;
  if (rows * prm->head_dim >= 9.0e18 || double(prm->batch) * prm->seqlen >= 2147483647.0 ||
      rows >= 2147483647.0)
    return fail(SA_ERR_UNSUPPORTED, "problem too large for 32-bit row indices");
  return SA_OK;
}

static sa_status_t check_ptrs(const void* q, const void* k, const void* v, const void* out) {
  if (!q || !k || !v || !out) return fail(SA_ERR_INVALID_ARG, "q, k, v and out must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(SA_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
  if (out == q || out == k || out == v) return fail(SA_ERR_INVALID_ARG, "out aliases an input");
  return SA_OK;
}

static Problem make_problem(const sa_params_t* prm, const void* q, const void* k, const void* v,
                            const int32_t* perm, void* out) {
  Problem pb{};
  pb.B = prm->batch;
  pb.n = prm->seqlen;
  pb.Hq = prm->num_q_heads;
  pb.Hkv = prm->num_kv_heads;
  pb.d = prm->head_dim;
  pb.g = pb.Hq / pb.Hkv;
  pb.window = prm->window;
  pb.window_swa = prm->window_swa > 0 ? prm->window_swa : prm->window;
  pb.causal = prm->causal ? 1 : 0;
  pb.scale = prm->softmax_scale > 0.f ? prm->softmax_scale : 1.0f / std::sqrt(float(pb.d));
  pb.q = q;
  pb.k = k;
  pb.v = v;
  pb.perm = perm;
  pb.out = out;
  pb.err = prm->err ? prm->err : default_error_word();
  return pb;
}

static sa_status_t finish_bwd(sa_status_t st, int32_t launches) {
  if (st == SA_OK) {
    g_last_launches = launches;
    g_msg[0] = '\0';
  }
  return st;
}

static sa_status_t finish(sa_status_t st, int32_t kernel, int32_t launches) {
  if (st == SA_OK) {
    g_last_kernel = kernel;
    g_last_launches = launches;
    g_msg[0] = '\0';
  }
  return st;
}

// The concrete kernel a request maps to for one path (SIMT, gather, ring,
// chunk), or 0 when the requested tcgen05 variant cannot run this shape.
// The tcgen05 preference: the ring kernel (narrow spans), else the chunk
// kernel (any span), else the gather kernel.
static int32_t pick_kernel(const sa_params_t* prm, const Problem& pb, Path path) {
  const bool ring = ring_supported(pb, path);
  const bool chunk = chunk_supported(pb, path);
  const bool gather = tc_supported(pb, path);
  const int32_t best = ring ? SA_KERNEL_TCGEN05_RING
                       : chunk ? SA_KERNEL_TCGEN05_CHUNK
                       : gather ? SA_KERNEL_TCGEN05_GATHER
                                : 0;
  switch (prm->kernel) {
    case SA_KERNEL_SIMT: return SA_KERNEL_SIMT;
    case SA_KERNEL_TCGEN05_RING: return ring ? SA_KERNEL_TCGEN05_RING : 0;
    case SA_KERNEL_TCGEN05_GATHER: return gather ? SA_KERNEL_TCGEN05_GATHER : 0;
    case SA_KERNEL_TCGEN05_CHUNK: return chunk ? SA_KERNEL_TCGEN05_CHUNK : 0;
    case SA_KERNEL_TCGEN05: return best;
    default: return best ? best : SA_KERNEL_SIMT;
  }
}

static sa_status_t launch_kernel(int32_t kernel, const Problem& pb, Path path, const float* gate,
                                 int accumulate, cudaStream_t s) {
  if (kernel == SA_KERNEL_TCGEN05_RING) return launch_ring(pb, path, gate, accumulate, s);
  if (kernel == SA_KERNEL_TCGEN05_CHUNK) return launch_chunk(pb, path, gate, accumulate, s);
  return launch_tc(pb, path, gate, accumulate, s);
}

// Runs one single-path attention (SA or SWA) with the requested kernel.
static sa_status_t run_single(const sa_params_t* prm, Problem& pb, Path path, cudaStream_t s) {
  if (pb.err == nullptr) return fail(SA_ERR_CUDA, "cannot resolve the library error word");
  const int32_t kernel = pick_kernel(prm, pb, path);
  if (kernel == 0)
    return fail(SA_ERR_UNSUPPORTED, "shape does not fit the requested tcgen05 kernel (window "
                "too wide, Hq/Hkv does not divide 128, or a device without tcgen05)");
  if (kernel == SA_KERNEL_SIMT) return finish(launch_simt(pb, path, s), SA_KERNEL_SIMT, 1);
  return finish(launch_kernel(kernel, pb, path, nullptr, 0, s), kernel, 1);
}

}  // namespace sa

using namespace sa;

extern "C" sa_status_t sa_forward(const sa_params_t* params, const void* q, const void* k,
                                  const void* v, const int32_t* perm, void* out,
                                  cudaStream_t stream) {
  sa_status_t st = check_params(params, true);
  if (st != SA_OK) return st;
  if ((st = check_ptrs(q, k, v, out)) != SA_OK) return st;
  if (perm == nullptr) return fail(SA_ERR_INVALID_ARG, "perm must be non-NULL");
  Problem pb = make_problem(params, q, k, v, perm, out);
  return run_single(params, pb, kPathSA, stream);
}

extern "C" sa_status_t swa_forward(const sa_params_t* params, const void* q, const void* k,
                                   const void* v, void* out, cudaStream_t stream) {
  sa_status_t st = check_params(params, true);
  if (st != SA_OK) return st;
  if ((st = check_ptrs(q, k, v, out)) != SA_OK) return st;
  Problem pb = make_problem(params, q, k, v, nullptr, out);
  pb.window_swa = params->window;
  return run_single(params, pb, kPathSWA, stream);
}

extern "C" size_t sa_gated_workspace_size(const sa_params_t*) { return 0; }

extern "C" sa_status_t sa_swa_gated_forward(const sa_params_t* params, const void* q,
                                            const void* k, const void* v, const int32_t* perm,
                                            const float* gate_sa_logits,
                                            const float* gate_swa_logits, void* out,
                                            void* workspace, size_t workspace_bytes,
                                            cudaStream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  sa_status_t st = check_params(params, true);
  if (st != SA_OK) return st;
  if ((st = check_ptrs(q, k, v, out)) != SA_OK) return st;
  if (!perm || !gate_sa_logits || !gate_swa_logits)
    return fail(SA_ERR_INVALID_ARG, "perm and both gate logit arrays must be non-NULL");
  Problem pb = make_problem(params, q, k, v, perm, out);
  pb.gate_sa = gate_sa_logits;
  pb.gate_swa = gate_swa_logits;
  if (pb.err == nullptr) return fail(SA_ERR_CUDA, "cannot resolve the library error word");
  const int32_t k_swa = pick_kernel(params, pb, kPathSWA);
  const int32_t k_sa = pick_kernel(params, pb, kPathSA);
  if (k_swa == 0 || k_sa == 0)
    return fail(SA_ERR_UNSUPPORTED, "shape does not fit the requested tcgen05 kernel");
  if (k_swa != SA_KERNEL_SIMT && k_sa != SA_KERNEL_SIMT) {
    // Pass 1 writes sigmoid(a_swa) * Y_swa into out; pass 2 adds
    // sigmoid(a_sa) * Y_sa row by row.  Stream order separates the passes and
    // sigma being a bijection means each pass writes each row exactly once.
    st = launch_kernel(k_swa, pb, kPathSWA, pb.gate_swa, 0, stream);
    if (st != SA_OK) return st;
    return finish(launch_kernel(k_sa, pb, kPathSA, pb.gate_sa, 1, stream), k_sa, 2);
  }
  return finish(launch_simt(pb, kPathGated, stream), SA_KERNEL_SIMT, 1);
}

// ------------------------------------------------------------------ backward

namespace sa {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace of one backward path: the rows' log2 normaliser and D (fp32).
static size_t rows_bytes(const sa_params_t* p) {
  return align256(size_t(p->batch) * p->seqlen * p->num_q_heads * sizeof(float));
}

static size_t gated_bwd_bytes(const sa_params_t* p) {
  const size_t tok = size_t(p->batch) * p->seqlen * p->head_dim;
  return 2 * rows_bytes(p) + align256(tok * p->num_q_heads * 4) +
         2 * align256(tok * p->num_kv_heads * 4);
}

static sa_status_t check_bwd(const sa_params_t* prm, const void* dout, const void* dq,
                             const void* dk, const void* dv, const void* q, const void* k,
                             const void* v, void* ws, size_t ws_bytes, size_t need) {
  if (!dout || !dq || !dk || !dv) return fail(SA_ERR_INVALID_ARG, "dout, dq, dk and dv must be non-NULL");
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(SA_ERR_INVALID_ARG, "dout, dq, dk and dv must be 16-byte aligned");
  const void* outs[3] = {dq, dk, dv};
  const void* ins[4] = {q, k, v, dout};
  for (const void* o : outs)
    for (const void* i : ins)
      if (o == i) return fail(SA_ERR_INVALID_ARG, "a gradient output aliases an input");
  if (dq == dk || dq == dv || dk == dv) return fail(SA_ERR_INVALID_ARG, "dq, dk and dv must differ");
  if (ws_bytes < need || ws == nullptr)
    return fail(SA_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu)", need, ws_bytes);
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(SA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (prm->kernel != SA_KERNEL_AUTO && prm->kernel != SA_KERNEL_TCGEN05)
    return fail(SA_ERR_UNSUPPORTED, "the backward pass runs on its tcgen05 kernels only");
  return SA_OK;
}

static sa_status_t run_bwd_single(const sa_params_t* params, const void* q, const void* k,
                                  const void* v, const int32_t* perm, const void* dout, void* dq,
                                  void* dk, void* dv, void* ws, size_t ws_bytes, Path path,
                                  cudaStream_t stream) {
  sa_status_t st = check_params(params, true);
  if (st != SA_OK) return st;
  if ((st = check_ptrs(q, k, v, dq)) != SA_OK) return st;
  if (path == kPathSA && perm == nullptr) return fail(SA_ERR_INVALID_ARG, "perm must be non-NULL");
  const size_t rb = rows_bytes(params);
  if ((st = check_bwd(params, dout, dq, dk, dv, q, k, v, ws, ws_bytes, 2 * rb)) != SA_OK) return st;
  Problem pb = make_problem(params, q, k, v, perm, dq);
  if (path == kPathSWA) pb.window_swa = params->window;
  if (pb.err == nullptr) return fail(SA_ERR_CUDA, "cannot resolve the library error word");
  if (!bwd_supported(pb, path))
    return fail(SA_ERR_UNSUPPORTED, "the backward kernels need d in {64, 128}, Hq/Hkv dividing 128, "
                "a key span of at most 256 per 128-row tile, and an sm_103 device");
  BwdArgs a{};
  a.dout = dout;
  a.lse2 = static_cast<float*>(ws);
  a.dsum = reinterpret_cast<float*>(static_cast<char*>(ws) + rb);
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.out_mode = 0;
  return finish_bwd(launch_bwd(pb, path, a, stream), 2);
}

}  // namespace sa

extern "C" size_t sa_backward_workspace_size(const sa_params_t* params) {
  if (params == nullptr || params->batch < 1 || params->seqlen < 1 || params->num_q_heads < 1)
    return 0;
  return 2 * rows_bytes(params);
}

extern "C" size_t sa_swa_gated_backward_workspace_size(const sa_params_t* params) {
  if (params == nullptr || params->batch < 1 || params->seqlen < 1 || params->num_q_heads < 1 ||
      params->num_kv_heads < 1 || params->head_dim < 1)
    return 0;
  return gated_bwd_bytes(params);
}

extern "C" sa_status_t sa_backward(const sa_params_t* params, const void* q, const void* k,
                                   const void* v, const int32_t* perm, const void* dout, void* dq,
                                   void* dk, void* dv, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream) {
  return run_bwd_single(params, q, k, v, perm, dout, dq, dk, dv, workspace, workspace_bytes,
                        kPathSA, stream);
}

extern "C" sa_status_t swa_backward(const sa_params_t* params, const void* q, const void* k,
                                    const void* v, const void* dout, void* dq, void* dk, void* dv,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return run_bwd_single(params, q, k, v, nullptr, dout, dq, dk, dv, workspace, workspace_bytes,
                        kPathSWA, stream);
}

// ------------------------------------------------------------------ backward, no allocation

namespace sa {

// Scratch of sa_backward_noalloc: the per-row log2 normaliser and D of the
// backward kernels (two fp32 values per (token, query head)), for at most
// kNoallocMaxRows rows, i.e. 8 MiB.  A file-scope device array: every device
// that loads this library holds it until the process exits.
constexpr size_t kNoallocMaxRows = size_t(1) << 20;
static __device__ __align__(256) float g_noalloc_scratch[2 * kNoallocMaxRows];

// The array's device address on each device, looked up once per device with
// that device current (in host code the array's name is only a stand-in).
constexpr int kNoallocMaxDevices = 64;
static std::mutex g_noalloc_mu;
static float* g_noalloc_ptr[kNoallocMaxDevices] = {};

static sa_status_t noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
  if (dev < 0 || dev >= kNoallocMaxDevices)
    return fail(SA_ERR_UNSUPPORTED, "device index %d beyond the %d this entry point tracks", dev,
                kNoallocMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    ce = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (ce != cudaSuccess || p == nullptr)
      return fail(SA_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s",
                  cudaGetErrorString(ce));
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return SA_OK;
}

}  // namespace sa

extern "C" sa_status_t sa_backward_noalloc(const sa_params_t* params, const void* q,
                                           const void* k, const void* v, const int32_t* perm,
                                           const void* dout, void* dq, void* dk, void* dv,
                                           cudaStream_t stream) {
  sa_status_t st = check_params(params, true);
  if (st != SA_OK) return st;
  const size_t rows = size_t(params->batch) * params->seqlen * params->num_q_heads;
  if (rows > kNoallocMaxRows)
    return fail(SA_ERR_UNSUPPORTED,
                "sa_backward_noalloc: batch * seqlen * num_q_heads = %zu exceeds the %zu rows "
                "its static scratch holds; use sa_backward with a workspace",
                rows, kNoallocMaxRows);
  float* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != SA_OK) return st;
  // Both halves are written for every row before they are read within the
  // call, so nothing needs clearing between calls.
  return run_bwd_single(params, q, k, v, perm, dout, dq, dk, dv, scratch,
                        2 * kNoallocMaxRows * sizeof(float), kPathSA, stream);
}

extern "C" sa_status_t sa_swa_gated_backward(const sa_params_t* params, const void* q,
                                             const void* k, const void* v, const int32_t* perm,
                                             const float* gate_sa_logits,
                                             const float* gate_swa_logits, const void* dout,
                                             void* dq, void* dk, void* dv, float* dgate_sa,
                                             float* dgate_swa, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream) {
  sa_status_t st = check_params(params, true);
  if (st != SA_OK) return st;
  if ((st = check_ptrs(q, k, v, dq)) != SA_OK) return st;
  if (!perm || !gate_sa_logits || !gate_swa_logits)
    return fail(SA_ERR_INVALID_ARG, "perm and both gate logit arrays must be non-NULL");
  const size_t need = gated_bwd_bytes(params);
  if ((st = check_bwd(params, dout, dq, dk, dv, q, k, v, workspace, workspace_bytes, need)) != SA_OK)
    return st;
  Problem pb = make_problem(params, q, k, v, perm, dq);
  if (pb.err == nullptr) return fail(SA_ERR_CUDA, "cannot resolve the library error word");
  if (!bwd_supported(pb, kPathSA) || !bwd_supported(pb, kPathSWA))
    return fail(SA_ERR_UNSUPPORTED, "the backward kernels need d in {64, 128}, Hq/Hkv dividing 128, "
                "a key span of at most 256 per 128-row tile, and an sm_103 device");
  const size_t rb = rows_bytes(params);
  const size_t tok = size_t(params->batch) * params->seqlen * params->head_dim;
  char* w = static_cast<char*>(workspace);
  float* dq32 = reinterpret_cast<float*>(w + 2 * rb);
  float* dk32 = reinterpret_cast<float*>(w + 2 * rb + align256(tok * params->num_q_heads * 4));
  float* dv32 = reinterpret_cast<float*>(reinterpret_cast<char*>(dk32) +
                                         align256(tok * params->num_kv_heads * 4));
  BwdArgs a{};
  a.dout = dout;
  a.lse2 = reinterpret_cast<float*>(w);
  a.dsum = reinterpret_cast<float*>(w + rb);
  a.dq = dq32;
  a.dk = dk32;
  a.dv = dv32;
  // SA path with its gate: stores; SWA path with its gate: adds.
  a.gate = gate_sa_logits;
  a.dgate = dgate_sa;
  a.out_mode = 1;
  if ((st = launch_bwd(pb, kPathSA, a, stream)) != SA_OK) return st;
  a.gate = gate_swa_logits;
  a.dgate = dgate_swa;
  a.out_mode = 2;
  if ((st = launch_bwd(pb, kPathSWA, a, stream)) != SA_OK) return st;
  if ((st = launch_to_bf16(dq32, dq, tok * params->num_q_heads, stream)) != SA_OK) return st;
  if ((st = launch_to_bf16(dk32, dk, tok * params->num_kv_heads, stream)) != SA_OK) return st;
  if ((st = launch_to_bf16(dv32, dv, tok * params->num_kv_heads, stream)) != SA_OK) return st;
  return finish_bwd(SA_OK, 7);
}

extern "C" sa_status_t sa_gate_projection(const void* x, int32_t tokens, int32_t d_model,
                                          int32_t num_q_heads, const void* w_sa,
                                          const void* w_swa, const float* b_sa,
                                          const float* b_swa, float* gate_sa_logits,
                                          float* gate_swa_logits, int32_t* d_err,
                                          cudaStream_t stream) {
  if (!x || !w_sa || !w_swa || !gate_sa_logits || !gate_swa_logits)
    return fail(SA_ERR_INVALID_ARG, "x, both weights and both logit outputs must be non-NULL");
  if (tokens < 1 || num_q_heads < 1 || d_model < 1)
    return fail(SA_ERR_INVALID_ARG, "tokens, d_model and num_q_heads must be >= 1");
  if (d_model % 64 != 0 || num_q_heads > 128)
    return fail(SA_ERR_UNSUPPORTED, "d_model must be a multiple of 64 and num_q_heads <= 128");
  if (!aligned16(x) || !aligned16(w_sa) || !aligned16(w_swa))
    return fail(SA_ERR_INVALID_ARG, "x and the weights must be 16-byte aligned");
  if (double(tokens) * d_model >= 9.0e18 || double(tokens) * num_q_heads >= 2147483647.0)
    return fail(SA_ERR_UNSUPPORTED, "problem too large");
  int32_t* err = d_err ? d_err : default_error_word();
  if (!err) return fail(SA_ERR_CUDA, "cannot resolve the library error word");
  sa_status_t st = launch_gate_projection(x, tokens, d_model, num_q_heads, w_sa, w_swa, b_sa, b_swa,
                                          gate_sa_logits, gate_swa_logits, err, stream);
  if (st == SA_OK) g_msg[0] = '\0';
  return st;
}

extern "C" sa_status_t sa_rope(void* x, int32_t batch, int32_t seqlen, int32_t heads,
                               int32_t head_dim, double base, cudaStream_t stream) {
  if (!x) return fail(SA_ERR_INVALID_ARG, "x must be non-NULL");
  if (batch < 1 || seqlen < 1 || heads < 1 || head_dim < 2 || head_dim % 2 != 0 || head_dim > 128)
    return fail(SA_ERR_INVALID_ARG, "need batch, seqlen, heads >= 1 and an even head_dim <= 128");
  if (!(base > 1.0)) return fail(SA_ERR_INVALID_ARG, "base must be > 1");
  if (double(batch) * seqlen >= 2147483647.0) return fail(SA_ERR_UNSUPPORTED, "batch * seqlen too large");
  sa_status_t st = launch_rope(x, batch, seqlen, heads, head_dim, base, stream);
  if (st == SA_OK) g_msg[0] = '\0';
  return st;
}

extern "C" size_t sa_receptive_field_workspace_size(int32_t n) {
  return n < 1 ? 0 : receptive_field_workspace_bytes(n);
}

extern "C" sa_status_t sa_receptive_field(const int32_t* perms, int32_t layers, int32_t n,
                                          int32_t window, int32_t causal, const int32_t* targets,
                                          int32_t num_targets, int64_t* sizes, void* workspace,
                                          size_t workspace_bytes, int32_t* d_err,
                                          cudaStream_t stream) {
  if (!perms || !targets || !sizes || !workspace)
    return fail(SA_ERR_INVALID_ARG, "perms, targets, sizes and workspace must be non-NULL");
  if (layers < 1 || layers > 64 || n < 1 || window < 1 || num_targets < 1)
    return fail(SA_ERR_INVALID_ARG, "need 1 <= layers <= 64, n >= 1, window >= 1, num_targets >= 1");
  if (workspace_bytes < receptive_field_workspace_bytes(n))
    return fail(SA_ERR_INVALID_ARG, "workspace of %zu bytes needed", receptive_field_workspace_bytes(n));
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0 || (reinterpret_cast<uintptr_t>(sizes) & 7u) != 0)
    return fail(SA_ERR_INVALID_ARG, "workspace must be 16-byte and sizes 8-byte aligned");
  int32_t* err = d_err ? d_err : default_error_word();
  if (!err) return fail(SA_ERR_CUDA, "cannot resolve the library error word");
  sa_status_t st = launch_receptive_field(perms, layers, n, window, causal ? 1 : 0, targets,
                                          num_targets, sizes, workspace, err, stream);
  if (st == SA_OK) g_msg[0] = '\0';
  return st;
}

extern "C" sa_status_t sa_inverse_perm(const int32_t* perm, int32_t* inv, int32_t batch,
                                       int32_t n, int32_t* d_err, cudaStream_t stream) {
  if (!perm || !inv) return fail(SA_ERR_INVALID_ARG, "perm and inv must be non-NULL");
  if (batch < 1 || n < 1) return fail(SA_ERR_INVALID_ARG, "batch and n must be >= 1");
  if (double(batch) * n >= 2147483647.0) return fail(SA_ERR_UNSUPPORTED, "batch * n too large");
  const int32_t* a = perm;
  const int32_t* b = inv;
  if (a < b + size_t(batch) * n && b < a + size_t(batch) * n)
    return fail(SA_ERR_INVALID_ARG, "perm and inv overlap");
  int32_t* err = d_err ? d_err : default_error_word();
  if (!err) return fail(SA_ERR_CUDA, "cannot resolve the library error word");
  sa_status_t st = launch_inverse_perm(perm, inv, batch, n, err, stream);
  if (st == SA_OK) g_msg[0] = '\0';
  return st;
}

extern "C" sa_status_t sa_make_perm(uint64_t seed, int32_t layer, int32_t batch_index, int32_t n,
                                    int32_t* perm_host) {
  if (!perm_host) return fail(SA_ERR_INVALID_ARG, "perm_host must be non-NULL");
  if (n < 1 || layer < 0 || batch_index < 0)
    return fail(SA_ERR_INVALID_ARG, "n must be >= 1; layer and batch_index >= 0");
  // splitmix64 (S. Vigna, public domain): add the golden-ratio increment, then
  // two xor-shift-multiply rounds and a final xor-shift.
  auto step = [](uint64_t& state) -> uint64_t {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  };
  uint64_t start = seed + (uint64_t(uint32_t(layer)) << 32) + uint64_t(uint32_t(batch_index));
  uint64_t state = step(start);  // the first output seeds this stream
  for (int32_t p = 0; p < n; ++p) perm_host[p] = p;
  for (int32_t i = n - 1; i >= 1; --i) {
    const uint64_t x = step(state);
    const uint64_t j = uint64_t((unsigned __int128)x * (unsigned __int128)(uint64_t(i) + 1) >> 64);
    const int32_t t = perm_host[i];
    perm_host[i] = perm_host[j];
    perm_host[j] = t;
  }
  g_msg[0] = '\0';
  return SA_OK;
}

extern "C" sa_status_t sa_check_error(const int32_t* d_err, cudaStream_t stream) {
  const int32_t* err = d_err ? d_err : default_error_word();
  if (!err) return fail(SA_ERR_CUDA, "cannot resolve the library error word");
  int32_t host = 0;
  cudaError_t ce = cudaMemcpyAsync(&host, err, sizeof(host), cudaMemcpyDeviceToHost, stream);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(stream);
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(ce));
  if (host & SA_ERRBIT_INTERNAL)
    return fail(SA_ERR_INTERNAL, "a device self-check of an internal index failed");
  if (host & SA_ERRBIT_TIMEOUT) return fail(SA_ERR_TIMEOUT, "a device wait ran past its bound");
  if (host & (SA_ERRBIT_RANGE | SA_ERRBIT_DUP))
    return fail(SA_ERR_BAD_PERM, "perm is not a permutation (error bits 0x%x)", host);
  return SA_OK;
}

extern "C" sa_status_t sa_clear_error(int32_t* d_err, cudaStream_t stream) {
  int32_t* err = d_err ? d_err : default_error_word();
  if (!err) return fail(SA_ERR_CUDA, "cannot resolve the library error word");
  cudaError_t ce = cudaMemsetAsync(err, 0, sizeof(int32_t), stream);
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "clearing the error word: %s", cudaGetErrorString(ce));
  return SA_OK;
}

extern "C" sa_status_t sa_set_wait_limit(int64_t cycles) {
  g_wait_limit.store(cycles > 0 ? (long long)cycles : kDefaultWaitLimit, std::memory_order_relaxed);
  g_msg[0] = '\0';
  return SA_OK;
}

extern "C" int64_t sa_get_wait_limit(void) { return wait_limit_cycles(); }

extern "C" const char* sa_status_string(sa_status_t status) {
  switch (status) {
    case SA_OK: return "SA_OK";
    case SA_ERR_INVALID_ARG: return "SA_ERR_INVALID_ARG: invalid argument";
    case SA_ERR_UNSUPPORTED: return "SA_ERR_UNSUPPORTED: not supported by this library";
    case SA_ERR_CUDA: return "SA_ERR_CUDA: CUDA runtime error";
    case SA_ERR_BAD_PERM: return "SA_ERR_BAD_PERM: perm is not a permutation";
    case SA_ERR_TIMEOUT: return "SA_ERR_TIMEOUT: device wait ran past its bound";
    case SA_ERR_INTERNAL: return "SA_ERR_INTERNAL: device self-check failed";
  }
  return "unknown sa_status_t";
}

extern "C" const char* sa_last_error_message(void) { return g_msg; }
extern "C" int32_t sa_last_kernel(void) { return g_last_kernel; }
extern "C" int32_t sa_last_launch_count(void) { return g_last_launches; }
