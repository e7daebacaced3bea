// CUDA-core SA / SWA / gated kernel: the correctness baseline, and the path
// for windows the tensor-core kernel does not take.
//
// One warp computes one output row (b, token, query head):
//   * SA ("Core mechanism" steps 1-3 of the Stochastic Attention summary):
//     the warp owns permuted position p, query token i = sigma[p]; its keys
//     are the tokens sigma[q] for |q - p| <= h (h = w/2, clipped to [0, n));
//     causal keeps only sigma[q] <= i; the result is written to row i (the
//     sigma^{-1} scatter).
//   * SWA ("Problem statement"): query token i = p, keys [max(0,i-w+1), i].
//   * gated ("Gated SA and SWA" equation): both windows for the same query,
//     merged as sigmoid(a_sa) * Y_sa + sigmoid(a_swa) * Y_swa in registers.
// Keys are taken 32 at a time: lane c computes the score of key c (a full
// d-long dot product against the query held in shared memory), the warp
// does an online-softmax update, and then the valid keys are accumulated
// into the output with each lane owning d/32 output elements (coalesced V
// row reads).  fp32 accumulation throughout; bf16 in and out.
#include <cuda_bf16.h>

#include <cmath>

#include "sa_internal.h"

namespace sa {
namespace {

struct SimtArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* perm;
  const float* gate_sa;
  const float* gate_swa;
  __nv_bfloat16* out;
  int B, n, Hq, Hkv, g;
  int h;       // SA half-width
  int w_swa;   // SWA window
  int causal;
  int path;
  float scale_log2;  // softmax scale * log2(e): scores are kept in log2 units
  int32_t* err;
};

constexpr int kWarps = 8;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int D>
struct RowState {
  float m = -INFINITY;  // running max (log2 units)
  float l = 0.f;        // this lane's share of the running denominator
  float acc[D / 32] = {};
};

// Online-softmax accumulation of one window.  key_of(c, j, valid) names the
// c-th candidate key token j of the window and whether it is attended.
template <int D, class KeyFn>
__device__ __forceinline__ void attend(const SimtArgs& a, const float* qs, int b, int kvh,
                                       int count, KeyFn key_of, RowState<D>& st) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const size_t tok_stride = size_t(a.Hkv) * D;
  const __nv_bfloat16* kb = a.k + size_t(b) * a.n * tok_stride + size_t(kvh) * D;
  const __nv_bfloat16* vb = a.v + size_t(b) * a.n * tok_stride + size_t(kvh) * D;
  for (int c0 = 0; c0 < count; c0 += 32) {
    const int c = c0 + lane;
    int j = 0;
    bool valid = false;
    if (c < count) key_of(c, j, valid);
    float s = -INFINITY;
    if (valid) {
      const uint4* kr = reinterpret_cast<const uint4*>(kb + size_t(j) * tok_stride);
      float dot = 0.f;
#pragma unroll
      for (int u = 0; u < D / 8; ++u) {
        const uint4 w4 = __ldg(kr + u);
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&w4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h2[e]);
          dot = fmaf(qs[u * 8 + 2 * e], f.x, dot);
          dot = fmaf(qs[u * 8 + 2 * e + 1], f.y, dot);
        }
      }
      s = dot;
    }
    const float bmax = warp_max(s);
    if (bmax == -INFINITY) continue;  // nothing attended in this group
    const float m_new = fmaxf(st.m, bmax);
    const float corr = exp2f(st.m - m_new);
    st.l *= corr;
#pragma unroll
    for (int e = 0; e < E; ++e) st.acc[e] *= corr;
    const float pr = valid ? exp2f(s - m_new) : 0.f;
    st.l += pr;
    st.m = m_new;
    unsigned vm = __ballot_sync(0xffffffffu, valid);
    while (vm) {
      const int t = __ffs(vm) - 1;
      vm &= vm - 1;
      const float pt = __shfl_sync(0xffffffffu, pr, t);
      const int jt = __shfl_sync(0xffffffffu, j, t);
      const __nv_bfloat16* vr = vb + size_t(jt) * tok_stride + lane * E;
      if constexpr (E == 4) {
        const uint2 w2 = __ldg(reinterpret_cast<const uint2*>(vr));
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w2.x));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w2.y));
        st.acc[0] = fmaf(pt, f0.x, st.acc[0]);
        st.acc[1] = fmaf(pt, f0.y, st.acc[1]);
        st.acc[2] = fmaf(pt, f1.x, st.acc[2]);
        st.acc[3] = fmaf(pt, f1.y, st.acc[3]);
      } else {
        const unsigned w1 = __ldg(reinterpret_cast<const unsigned*>(vr));
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w1));
        st.acc[0] = fmaf(pt, f0.x, st.acc[0]);
        st.acc[1] = fmaf(pt, f0.y, st.acc[1]);
      }
    }
  }
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + expf(-x)); }

template <int D>
__global__ void __launch_bounds__(kWarps * 32) sa_simt_kernel(const SimtArgs a) {
  constexpr int E = D / 32;
  __shared__ float qsm[kWarps][D];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kWarps + warp;
  const long long total = (long long)a.B * a.n * a.Hq;
  if (row >= total) return;  // warp-uniform
  const int hq = int(row % a.Hq);
  const long long bp = row / a.Hq;
  const int p = int(bp % a.n);
  const int b = int(bp / a.n);
  const int kvh = hq / a.g;
  const int32_t* pb = a.perm ? a.perm + size_t(b) * a.n : nullptr;
  int i = p;
  if (a.path != kPathSWA) {
    i = pb[p];
    if (i < 0 || i >= a.n) {
      if (lane == 0) atomicOr(a.err, SA_ERRBIT_RANGE);
      return;
    }
  }
  const size_t out_row = (size_t(b) * a.n + i) * a.Hq + hq;
  if (out_row >= size_t(total)) {  // never expected: record and skip
    if (lane == 0) atomicOr(a.err, SA_ERRBIT_INTERNAL);
    return;
  }
  const __nv_bfloat16* qr = a.q + out_row * D;
  float* qs = qsm[warp];
  for (int e = lane; e < D; e += 32) qs[e] = __bfloat162float(qr[e]) * a.scale_log2;
  __syncwarp();

  float y[E];
  RowState<D> sa_st, swa_st;
  if (a.path != kPathSWA) {
    const int lo = max(0, p - a.h);
    const int hi = min(a.n - 1, p + a.h);
    const int causal = a.causal;
    const int n = a.n;
    int32_t* err = a.err;
    attend<D>(a, qs, b, kvh, hi - lo + 1,
              [&](int c, int& j, bool& valid) {
                j = pb[lo + c];
                if (j < 0 || j >= n) {
                  atomicOr(err, SA_ERRBIT_RANGE);
                  j = 0;
                  valid = false;
                  return;
                }
                valid = !causal || j <= i;
              },
              sa_st);
  }
  if (a.path != kPathSA) {
    const int lo = max(0, i - a.w_swa + 1);
    attend<D>(a, qs, b, kvh, i - lo + 1,
              [&](int c, int& j, bool& valid) {
                j = lo + c;
                valid = true;
              },
              swa_st);
  }
  if (a.path == kPathGated) {
    const float l1 = warp_sum(sa_st.l), l2 = warp_sum(swa_st.l);
    const float g1 = sigmoidf_(a.gate_sa[out_row]);
    const float g2 = sigmoidf_(a.gate_swa[out_row]);
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = g1 * (sa_st.acc[e] / l1) + g2 * (swa_st.acc[e] / l2);
  } else {
    const RowState<D>& st = (a.path == kPathSA) ? sa_st : swa_st;
    const float l = warp_sum(st.l);
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = st.acc[e] / l;
  }
  __nv_bfloat16* orow = a.out + out_row * D + lane * E;
  if constexpr (E == 4) {
    __nv_bfloat162 lo2 = __floats2bfloat162_rn(y[0], y[1]);
    __nv_bfloat162 hi2 = __floats2bfloat162_rn(y[2], y[3]);
    uint2 w2;
    w2.x = *reinterpret_cast<unsigned*>(&lo2);
    w2.y = *reinterpret_cast<unsigned*>(&hi2);
    *reinterpret_cast<uint2*>(orow) = w2;
  } else {
    __nv_bfloat162 v2 = __floats2bfloat162_rn(y[0], y[1]);
    *reinterpret_cast<__nv_bfloat162*>(orow) = v2;
  }
}

}  // namespace

sa_status_t launch_simt(const Problem& pb, Path path, cudaStream_t stream) {
  SimtArgs a;
  a.q = static_cast<const __nv_bfloat16*>(pb.q);
  a.k = static_cast<const __nv_bfloat16*>(pb.k);
  a.v = static_cast<const __nv_bfloat16*>(pb.v);
  a.perm = pb.perm;
  a.gate_sa = pb.gate_sa;
  a.gate_swa = pb.gate_swa;
  a.out = static_cast<__nv_bfloat16*>(pb.out);
  a.B = pb.B;
  a.n = pb.n;
  a.Hq = pb.Hq;
  a.Hkv = pb.Hkv;
  a.g = pb.g;
  a.h = pb.window / 2;
  a.w_swa = (path == kPathSWA) ? pb.window : pb.window_swa;
  a.causal = pb.causal;
  a.path = path;
  a.scale_log2 = pb.scale * 1.4426950408889634f;
  a.err = pb.err;
  const long long rows = (long long)pb.B * pb.n * pb.Hq;
  const unsigned blocks = unsigned((rows + kWarps - 1) / kWarps);
  if (pb.d == 128)
    sa_simt_kernel<128><<<blocks, kWarps * 32, 0, stream>>>(a);
  else
    sa_simt_kernel<64><<<blocks, kWarps * 32, 0, stream>>>(a);
  const cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "SIMT kernel launch: %s", cudaGetErrorString(ce));
  return SA_OK;
}

}  // namespace sa
