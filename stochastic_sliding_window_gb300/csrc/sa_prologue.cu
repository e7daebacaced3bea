// What feeds the attention paths: the two gate projections and the rotary
// position embedding by original token index.
//
// Gates ("Gated SA and SWA" section of the Stochastic Attention summary: the
// two paths are mixed through independent sigmoid projections).  The logits
// of both projections of the layer input come out of ONE tcgen05 GEMM,
//   [a_sa | a_swa] = x [W_sa ; W_swa]^T + [b_sa | b_swa],
// M = 128 tokens per tile, N = 2 Hq (padded to 32), K = d_model in 64-column
// blocks: x and both weight blocks are gathered with cp.async into
// double-buffered shared memory (128-byte swizzle) while the previous block's
// MMAs run; the bias is added in the epilogue and each token's two logit rows
// are written.  The sigmoid is applied where the paths merge (the attention
// epilogues), so the logits are what the gated calls take.
//
// RoPE before the gather: Q and K are rotated by each token's ORIGINAL index
// i (pairs (x_k, x_{k+d/2}) turned by i * theta_k, theta_k = base^(-2k/d)),
// so that a score depends on i - j whatever permutation brings the two
// tokens into one window.  One block per token; the angle is reduced to
// [-pi, pi] in fp64 before the fp32 sine and cosine, so positions in the
// hundreds of thousands keep their precision.
#include "sa_internal.h"
#include "sa_tc_common.cuh"

#include <cmath>
#include <cstring>

namespace sa {
namespace pro {

using namespace tcc;

constexpr int kThreads = 128;
constexpr int kKB = 64;  // d_model columns per block (128 bytes of bf16)
constexpr int kMaxStages = 4;

struct GateParams {
  const __nv_bfloat16* x;    // [M, D]
  const __nv_bfloat16* w_sa;  // [Hq, D]
  const __nv_bfloat16* w_swa;
  const float* b_sa;          // [Hq] or nullptr
  const float* b_swa;
  float* a_sa;                // [M, Hq]
  float* a_swa;
  int32_t* err;
  int M, D, Hq, n_pad, num_tiles;
  int stages;                          // x/w blocks in flight: 2 or kMaxStages (a power of two)
  uint32_t x_bytes, w_bytes, off_bar;  // one stage's x and w blocks; barrier offset
  long long timeout_cycles;
};

__global__ void __launch_bounds__(kThreads, 2) sa_gate_proj_kernel(const __grid_constant__ GateParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t stage_bytes = P.x_bytes + P.w_bytes;
  const uint32_t bars = sbase + P.off_bar;  // [kMaxStages] MMA of the stage done, then the drain
  const uint32_t drain_bar = bars + 8 * kMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P.off_bar + 8 * kMaxStages + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.off_bar + 8 * kMaxStages + 12);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int S = P.stages;
  const long long smask = S - 1;
  const int sshift = S == 4 ? 2 : 1;
  if (tid == 0) {
    for (int i = 0; i <= kMaxStages; ++i) mbar_init(bars + 8 * i, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // padded weight rows stay zero in every stage
  for (int st = 0; st < S; ++st)
    for (int i = 2 * P.Hq * 128 + tid * 16; i < P.n_pad * 128; i += kThreads * 16)
      *reinterpret_cast<uint4*>(smem + st * stage_bytes + P.x_bytes + i) = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(256u)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t trow = tmem + (uint32_t(warp * 32) << 16);
  const int nkb = P.D / kKB;
  const uint32_t id = idesc_bf16(kBM, P.n_pad, 0);
  // Blocks are numbered over all of this CTA's tiles: block g uses stage
  // g mod S, and its MMA commit completes phase g / S of that stage's barrier.
  long long g0 = 0;  // number of this CTA's first block in the current tile
  bool alive = true;
  for (int tile = blockIdx.x; tile < P.num_tiles && alive; tile += gridDim.x, g0 += nkb) {
    const int m0 = tile * kBM;
    // one 64-column block of x (128 rows) and of both weights (2 Hq rows)
    auto load = [&](int kb) {
      const uint32_t xs = sbase + uint32_t((g0 + kb) & smask) * stage_bytes, ws = xs + P.x_bytes;
      for (int idx = tid; idx < kBM * 8; idx += kThreads) {
        const int r = idx >> 3, c = idx & 7;
        const int m = min(m0 + r, P.M - 1);
        cp_async16(xs + r * 128 + ((c ^ (r & 7)) << 4), P.x + size_t(m) * P.D + kb * kKB + c * 8);
      }
      for (int idx = tid; idx < 2 * P.Hq * 8; idx += kThreads) {
        const int r = idx >> 3, c = idx & 7;
        const __nv_bfloat16* w = r < P.Hq ? P.w_sa + size_t(r) * P.D : P.w_swa + size_t(r - P.Hq) * P.D;
        cp_async16(ws + r * 128 + ((c ^ (r & 7)) << 4), w + kb * kKB + c * 8);
      }
    };
    // the first S - 1 blocks (their stages were last read by MMAs that the
    // previous tile's final wait covers); one commit group per block, empty
    // past the last block, so the group count stays uniform
    for (int j = 0; j < S - 1; ++j) {
      if (j < nkb) load(j);
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
    for (int kb = 0; kb < nkb; ++kb) {
      const long long gb = g0 + kb;
      const int nk = kb + S - 1;  // the block loaded now, into the stage block kb - 1 used
      if (nk < nkb) {
        if (kb >= 1) {
          const long long gp = gb - 1;
          const bool ok = bounded_wait(bars + 8 * uint32_t(gp & smask), uint32_t(gp >> sshift) & 1u,
                                       P.timeout_cycles, P.err, abort_flag);
          if (__syncthreads_or(ok ? 0 : 1)) {
            alive = false;
            break;
          }
        }
        load(nk);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      // groups committed so far: kb + S; at most S - 1 pending means block kb landed
      if (S == 4)
        asm volatile("cp.async.wait_group 3;" ::: "memory");
      else
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const uint32_t xs = sbase + uint32_t(gb & smask) * stage_bytes;
        const uint64_t a0 = sdesc_sw128(xs, 16, 1024), b0 = sdesc_sw128(xs + P.x_bytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kKB / 16; ++kk)
          umma_bf16(tmem, a0 + 2 * kk, b0 + 2 * kk, id, (kb > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bars + 8 * uint32_t(gb & smask));
      }
    }
    if (!alive) break;
    // the last block's MMAs (and with them all earlier ones) are done
    {
      const long long gl = g0 + nkb - 1;
      const bool ok = bounded_wait(bars + 8 * uint32_t(gl & smask), uint32_t(gl >> sshift) & 1u,
                                   P.timeout_cycles, P.err, abort_flag);
      if (__syncthreads_or(ok ? 0 : 1)) break;
    }
    tc_fence_after();
    const int m = m0 + tid;
    for (int c0 = 0; c0 < P.n_pad; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(trow + c0, v);  // every lane: the load is warp-collective
      if (m < P.M) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = c0 + e;
          if (col < P.Hq) {
            P.a_sa[size_t(m) * P.Hq + col] =
                __uint_as_float(v[e]) + (P.b_sa ? P.b_sa[col] : 0.f);
          } else if (col < 2 * P.Hq) {
            P.a_swa[size_t(m) * P.Hq + col - P.Hq] =
                __uint_as_float(v[e]) + (P.b_swa ? P.b_swa[col - P.Hq] : 0.f);
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();  // TMEM is overwritten by the next tile
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (tid == 0) {
    umma_commit(drain_bar);
    const long long t0 = clock64();
    while (!mbar_try_wait(drain_bar, 0) && clock64() - t0 < kDrainCycles) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256u)
                 : "memory");
  }
}

struct RopeParams {
  __nv_bfloat16* x;  // [B, n, H, d], rotated in place
  long long rows;    // B * n
  int n, H, d;
  int vec;           // 16-byte accesses: x 16-byte aligned and d/2 a multiple of 8
  int pairs;         // else 4-byte accesses: x 4-byte aligned and d/2 even (else 2-byte)
  int tpb;           // tokens per block on the 16-byte path
  double theta[64];  // base^(-2k/d), k < d/2
};

constexpr int kRopePre = 4;     // 16-byte items per thread loaded before the angles
constexpr int kRopeAngles = 512;  // angle slots per block (tokens per block x d/2)

// The angle i * theta_k of token i, reduced to [-pi, pi] in fp64, then its
// cosine and sine in fp32.
__device__ __forceinline__ void rope_angle(const RopeParams& P, long long row, int k, float& c,
                                           float& s) {
  const double a = double(row % P.n) * P.theta[k];
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  sincosf(float(a - two_pi * rint(a * inv_two_pi)), &s, &c);
}

// 8 rotated pairs: (lo_e, hi_e) -> (lo_e c - hi_e s, hi_e c + lo_e s).
__device__ __forceinline__ void rope_rotate8(uint4& lo, uint4& hi, const float* cs, const float* sn) {
  uint32_t* pl = reinterpret_cast<uint32_t*>(&lo);
  uint32_t* ph = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __nv_bfloat162 bl = *reinterpret_cast<__nv_bfloat162*>(&pl[e]);
    __nv_bfloat162 bh = *reinterpret_cast<__nv_bfloat162*>(&ph[e]);
    const float2 l = __bfloat1622float2(bl), h = __bfloat1622float2(bh);
    const float c0 = cs[2 * e], s0 = sn[2 * e], c1 = cs[2 * e + 1], s1 = sn[2 * e + 1];
    bl = __floats2bfloat162_rn(l.x * c0 - h.x * s0, l.y * c1 - h.y * s1);
    bh = __floats2bfloat162_rn(h.x * c0 + l.x * s0, h.y * c1 + l.y * s1);
    pl[e] = *reinterpret_cast<uint32_t*>(&bl);
    ph[e] = *reinterpret_cast<uint32_t*>(&bh);
  }
}

__global__ void __launch_bounds__(kThreads) sa_rope_kernel(const __grid_constant__ RopeParams P) {
  __shared__ float s_cos[kRopeAngles], s_sin[kRopeAngles];
  const int half = P.d / 2;
  if (P.vec) {
    // tpb tokens per block; item = (token, head, 8 pairs).  The first items'
    // rows are loaded before the angles are computed, so the loads overlap
    // the fp64 angle reduction.
    const int h8 = half / 8;
    const int per_tok = P.H * h8;
    const long long row0 = (long long)blockIdx.x * P.tpb;
    const int ntok = int(min((long long)P.tpb, P.rows - row0));
    const int items = ntok * per_tok;
    uint4 vlo[kRopePre], vhi[kRopePre];
#pragma unroll
    for (int u = 0; u < kRopePre; ++u) {
      const int idx = threadIdx.x + u * kThreads;
      if (idx < items) {
        const int tk = idx / per_tok, rem = idx - tk * per_tok;
        const int h = rem / h8, k = (rem - h * h8) * 8;
        const __nv_bfloat16* px = P.x + (size_t(row0 + tk) * P.H + h) * P.d + k;
        vlo[u] = *reinterpret_cast<const uint4*>(px);
        vhi[u] = *reinterpret_cast<const uint4*>(px + half);
      }
    }
    for (int a = threadIdx.x; a < ntok * half; a += kThreads) {
      const int tk = a / half, k = a - tk * half;
      rope_angle(P, row0 + tk, k, s_cos[a], s_sin[a]);
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kRopePre; ++u) {
      const int idx = threadIdx.x + u * kThreads;
      if (idx < items) {
        const int tk = idx / per_tok, rem = idx - tk * per_tok;
        const int h = rem / h8, k = (rem - h * h8) * 8;
        __nv_bfloat16* px = P.x + (size_t(row0 + tk) * P.H + h) * P.d + k;
        rope_rotate8(vlo[u], vhi[u], s_cos + tk * half + k, s_sin + tk * half + k);
        *reinterpret_cast<uint4*>(px) = vlo[u];
        *reinterpret_cast<uint4*>(px + half) = vhi[u];
      }
    }
    for (int idx = threadIdx.x + kRopePre * kThreads; idx < items; idx += kThreads) {
      const int tk = idx / per_tok, rem = idx - tk * per_tok;
      const int h = rem / h8, k = (rem - h * h8) * 8;
      __nv_bfloat16* px = P.x + (size_t(row0 + tk) * P.H + h) * P.d + k;
      uint4 lo = *reinterpret_cast<const uint4*>(px), hi = *reinterpret_cast<const uint4*>(px + half);
      rope_rotate8(lo, hi, s_cos + tk * half + k, s_sin + tk * half + k);
      *reinterpret_cast<uint4*>(px) = lo;
      *reinterpret_cast<uint4*>(px + half) = hi;
    }
    return;
  }
  // one token per block, 4-byte or 2-byte accesses
  const long long row = blockIdx.x;  // (b, i)
  if (threadIdx.x < half) rope_angle(P, row, threadIdx.x, s_cos[threadIdx.x], s_sin[threadIdx.x]);
  __syncthreads();
  __nv_bfloat16* base = P.x + size_t(row) * P.H * P.d;
  if (P.pairs) {  // two adjacent pairs per thread, bf16x2 accesses
    const int h2 = half / 2;
    for (int idx = threadIdx.x; idx < P.H * h2; idx += blockDim.x) {
      const int h = idx / h2, k = 2 * (idx - (idx / h2) * h2);
      __nv_bfloat162* plo = reinterpret_cast<__nv_bfloat162*>(base + size_t(h) * P.d + k);
      __nv_bfloat162* phi = reinterpret_cast<__nv_bfloat162*>(base + size_t(h) * P.d + k + half);
      const float2 lo = __bfloat1622float2(*plo), hi = __bfloat1622float2(*phi);
      const float c0 = s_cos[k], s0 = s_sin[k], c1 = s_cos[k + 1], s1 = s_sin[k + 1];
      *plo = __floats2bfloat162_rn(lo.x * c0 - hi.x * s0, lo.y * c1 - hi.y * s1);
      *phi = __floats2bfloat162_rn(hi.x * c0 + lo.x * s0, hi.y * c1 + lo.y * s1);
    }
  } else {
    for (int idx = threadIdx.x; idx < P.H * half; idx += blockDim.x) {
      const int h = idx / half, k = idx - (idx / half) * half;
      __nv_bfloat16* px = base + size_t(h) * P.d;
      const float lo = __bfloat162float(px[k]), hi = __bfloat162float(px[k + half]);
      const float c = s_cos[k], s = s_sin[k];
      px[k] = __float2bfloat16_rn(lo * c - hi * s);
      px[k + half] = __float2bfloat16_rn(hi * c + lo * s);
    }
  }
}

}  // namespace pro

sa_status_t launch_gate_projection(const void* x, int tokens, int d_model, int hq, const void* w_sa,
                                   const void* w_swa, const float* b_sa, const float* b_swa,
                                   float* a_sa, float* a_swa, int32_t* err, cudaStream_t stream) {
  using namespace pro;
  int dev = 0, sms = 0, major = 0, minor = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3) return fail(SA_ERR_UNSUPPORTED, "device is not sm_103");
  GateParams P;
  std::memset(&P, 0, sizeof(P));
  P.x = static_cast<const __nv_bfloat16*>(x);
  P.w_sa = static_cast<const __nv_bfloat16*>(w_sa);
  P.w_swa = static_cast<const __nv_bfloat16*>(w_swa);
  P.b_sa = b_sa;
  P.b_swa = b_swa;
  P.a_sa = a_sa;
  P.a_swa = a_swa;
  P.err = err;
  P.M = tokens;
  P.D = d_model;
  P.Hq = hq;
  P.n_pad = (2 * hq + 31) / 32 * 32;
  P.num_tiles = (tokens + kBM - 1) / kBM;
  P.x_bytes = kBM * 128;
  P.w_bytes = uint32_t(P.n_pad) * 128;
  // four blocks in flight when two such CTAs fit an SM, else two
  const uint32_t stage_bytes = P.x_bytes + P.w_bytes;
  P.stages = uint32_t(kMaxStages) * stage_bytes <= 100u * 1024 ? kMaxStages : 2;
  P.off_bar = uint32_t(P.stages) * stage_bytes;
  P.timeout_cycles = wait_limit_cycles();
  // at least 80 KB per CTA: at most two CTAs share an SM, so their two
  // 256-column TMEM allocations always fit
  const uint32_t need = P.off_bar + 8 * (kMaxStages + 1) + 16 + 1024;
  const uint32_t smem = need > 80u * 1024 ? need : 80u * 1024;
  cudaError_t ce = cudaFuncSetAttribute(sa_gate_proj_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (ce == cudaSuccess) {
    // two CTAs per SM (256 TMEM columns each) so one's loads overlap the
    // other's MMAs and epilogue
    const int grid = P.num_tiles < 2 * sms ? P.num_tiles : 2 * sms;
    sa_gate_proj_kernel<<<grid, kThreads, smem, stream>>>(P);
    ce = cudaGetLastError();
  }
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "gate projection launch: %s", cudaGetErrorString(ce));
  return SA_OK;
}

sa_status_t launch_rope(void* x, int batch, int n, int heads, int head_dim, double base,
                        cudaStream_t stream) {
  using namespace pro;
  RopeParams P;
  std::memset(&P, 0, sizeof(P));
  P.x = static_cast<__nv_bfloat16*>(x);
  P.rows = (long long)batch * n;
  P.n = n;
  P.H = heads;
  P.d = head_dim;
  for (int k = 0; k < head_dim / 2; ++k) P.theta[k] = std::pow(base, -2.0 * k / head_dim);
  const int half = head_dim / 2;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(x);
  P.vec = (half % 8 == 0) && (addr % 16 == 0);
  P.pairs = (half % 2 == 0) && (addr % 4 == 0);
  unsigned grid = unsigned(P.rows);
  if (P.vec) {
    // enough tokens per block to give every thread an item, within the
    // block's angle slots
    const int per_tok = heads * (half / 8);
    int tpb = per_tok >= kThreads ? 1 : kThreads / per_tok;
    if (tpb * half > kRopeAngles) tpb = kRopeAngles / half;
    P.tpb = tpb < 1 ? 1 : tpb;
    grid = unsigned((P.rows + P.tpb - 1) / P.tpb);
  }
  sa_rope_kernel<<<grid, kThreads, 0, stream>>>(P);
  const cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "rope launch: %s", cudaGetErrorString(ce));
  return SA_OK;
}

}  // namespace sa
