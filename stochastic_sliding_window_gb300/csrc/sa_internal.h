// Internal interface between the C-ABI entry points (sa_api.cu) and the
// kernel launchers (sa_perm.cu, sa_simt.cu, sa_tc.cu, sa_tc_ring.cu,
// sa_tc_chunk.cu).  Not installed.
#pragma once

#include <cuda.h>  // CUtensorMap (type only)
#include <cuda_runtime.h>
#include <stdint.h>

#include "libsa.h"

namespace sa {

// Which attention a launch computes.
enum Path : int {
  kPathSA = 0,     // sliding window over the sigma-permuted rows
  kPathSWA = 1,    // trailing window over the original order
  kPathGated = 2,  // sigmoid-gated SA + SWA (SIMT kernel computes both in one pass)
};

// One attention problem, already validated on the host.
struct Problem {
  int B, n, Hq, Hkv, d, g;  // g = Hq / Hkv
  int window;               // SA window w (h = w / 2)
  int window_swa;           // SWA window
  int causal;               // SA causal rule
  float scale;              // softmax scale
  const void* q;
  const void* k;
  const void* v;
  const int32_t* perm;      // [B, n]; unused by SWA
  const float* gate_sa;     // [B, n, Hq] logits (gated only)
  const float* gate_swa;
  void* out;
  int32_t* err;             // device error word (never NULL here)
};

// Record a detail message for sa_last_error_message() and return `st`.
sa_status_t fail(sa_status_t st, const char* fmt, ...);

// Device error word owned by the library (used when the caller passes NULL).
int32_t* default_error_word();

// Bound, in SM cycles, on every pipeline wait of the tcgen05 kernels
// launched from now on (default ~2 s at the maximum clock; sa_set_wait_limit).
long long wait_limit_cycles();

// SIMT (CUDA-core) kernel: any window.  `path` selects SA, SWA or gated.
sa_status_t launch_simt(const Problem& pb, Path path, cudaStream_t stream);

// tcgen05 kernel.  `path` is kPathSA or kPathSWA.  gate != nullptr scales the
// output by sigmoid(gate logit); accumulate != 0 adds the previous contents
// of out (the gated merge's second pass).  Returns SA_ERR_UNSUPPORTED, with
// nothing launched, when the shape does not fit the kernel.
sa_status_t launch_tc(const Problem& pb, Path path, const float* gate, int accumulate,
                      cudaStream_t stream);

// True when launch_tc can run this problem / path.
bool tc_supported(const Problem& pb, Path path);

// tcgen05 kernel with a sliding K/V ring in shared memory (each CTA walks a
// contiguous run of tiles and fetches only the new rows of each window).
// Same contract as launch_tc; narrower spans only.
sa_status_t launch_ring(const Problem& pb, Path path, const float* gate, int accumulate,
                        cudaStream_t stream);
bool ring_supported(const Problem& pb, Path path);

// tcgen05 kernel streaming each tile's key span through shared memory in
// 128-key chunks with an online softmax: any window.  Same contract as
// launch_tc.
sa_status_t launch_chunk(const Problem& pb, Path path, const float* gate, int accumulate,
                         cudaStream_t stream);
bool chunk_supported(const Problem& pb, Path path);

// Tensor map of a row-major bf16 [rows, d] tensor for TMA copies of
// 64-column x box_rows boxes with the 128-byte swizzle (false if the driver
// entry point or the encoding fails).
bool encode_row_map(CUtensorMap* m, const void* base, uint64_t rows, int d, int box_rows);

// Backward pass (sa_bwd.cu).  One path (SA or SWA) per call: the dQ kernel
// over query tiles (writes the rows' log2 normaliser and D, and the
// gate-logit gradient when a gate is given), then the dK/dV kernel over
// 128-key tiles.  out_mode: 0 bf16 store, 1 fp32 store, 2 fp32 add.
struct BwdArgs {
  const void* dout;    // bf16 [B, n, Hq, d]
  const float* gate;   // [B, n, Hq] logits or nullptr
  float* lse2;         // [B, n, Hq] workspace
  float* dsum;         // [B, n, Hq] workspace
  float* dgate;        // [B, n, Hq] or nullptr
  void* dq;            // [B, n, Hq, d]
  void* dk;            // [B, n, Hkv, d]
  void* dv;
  int out_mode;
};
bool bwd_supported(const Problem& pb, Path path);
sa_status_t launch_bwd(const Problem& pb, Path path, const BwdArgs& a, cudaStream_t stream);
// fp32 -> bf16 conversion of `count` values (a multiple of 4).
sa_status_t launch_to_bf16(const float* src, void* dst, size_t count, cudaStream_t stream);

// Receptive fields of stacked SA layers (sa_graph.cu).
size_t receptive_field_workspace_bytes(int n);
sa_status_t launch_receptive_field(const int32_t* perms, int layers, int n, int window, int causal,
                                   const int32_t* targets, int num_targets, int64_t* sizes,
                                   void* workspace, int32_t* err, cudaStream_t s);

// The gate projections and RoPE (sa_prologue.cu).
sa_status_t launch_gate_projection(const void* x, int tokens, int d_model, int hq, const void* w_sa,
                                   const void* w_swa, const float* b_sa, const float* b_swa,
                                   float* a_sa, float* a_swa, int32_t* err, cudaStream_t stream);
sa_status_t launch_rope(void* x, int batch, int n, int heads, int head_dim, double base,
                        cudaStream_t stream);

// sigma^{-1} kernels.
sa_status_t launch_inverse_perm(const int32_t* perm, int32_t* inv, int batch, int n,
                                int32_t* err, cudaStream_t stream);

}  // namespace sa
