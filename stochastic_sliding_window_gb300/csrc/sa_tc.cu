// Tensor-core (tcgen05 / TMEM / TMA) kernel for SA and SWA on sm_103a.
//
// What one tile computes (Stochastic Attention summary, "Core mechanism"
// steps 1-3; causal rule from "Theoretical properties"; SWA from "Problem
// statement"):  a tile is Bt = 128/g consecutive PERMUTED positions
// p0 .. p0+Bt-1 of one (sequence b, kv head) pair, stacked with the g query
// heads that share that kv head, so the tile has M = 128 query rows
// (row r = t*g + j: position p0+t, query head kvh*g + j).  Their keys are the
// contiguous permuted span q in [p0 - left, p0 + Bt - 1 + right]
// (SA: left = right = h = w/2; SWA: left = w-1, right = 0, sigma = identity).
//
//   1. gather    (warp 0, TMA tile::gather4): sigma of the span -> smem; the
//                Q rows sigma[p0+t] and the K/V rows sigma[q] are fetched
//                straight from the BSHD tensors into 128B-swizzled smem --
//                the permuted copies never exist in HBM.
//   2. S = Q K^T (warp 1, tcgen05.mma kind::f16, fp32 accumulator in TMEM),
//                one 128 x span_pad tile: the whole window of every row.
//   3. softmax   (warps 4-11, two warpgroups taking alternate tiles; thread
//                r owns TMEM lane r): mask |p-q| <= h via the row's column
//                band, the sequence ends, and for causal SA sigma[q] <=
//                sigma[p]; exact row max, exp2, row sum; P (bf16) -> smem,
//                over the dead Q/K bytes.
//   4. O = P V   (warp 1, tcgen05.mma, V used MN-major), into the TMEM
//                columns S occupied.
//   5. epilogue  (same warpgroup): O / rowsum, optionally * sigmoid(gate)
//                and + the previous out row (the gated merge), bf16, stored
//                to out row sigma[p0+t] -- the sigma^{-1} scatter.
// Because one tile holds the whole window of each row there is no online
// rescaling.  The kernel is persistent (one CTA per SM, tiles strided by
// gridDim.x so neighbouring tiles -- which share halo K/V rows -- run at the
// same time and meet in L2).  Every mbarrier wait is bounded; on expiry the
// CTA sets SA_ERRBIT_TIMEOUT, drains its own copies and MMAs, frees TMEM and
// exits.
#include <cuda.h>  // CUtensorMap and the tensor-map enums (types only)
#include <cuda_bf16.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "sa_internal.h"
#include "sa_tc_common.cuh"

namespace sa {
namespace tc {

using namespace tcc;

constexpr int kThreads = 384;  // three warpgroups
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;  // also allocates and frees TMEM
constexpr int kTmemWarp = 1;
constexpr int kFirstSoftmaxWarp = 4;  // warpgroups 1 and 2 (warps 4-7, 8-11)
// Register split: launched at kLaunchRegs per thread (384 x 168 = 64512),
// warpgroup 0 (producer, MMA) gives registers back and the two softmax
// warpgroups take them: 128 x 64 + 256 x 216 = 63488 <= 64512.
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 64;
constexpr int kSoftmaxRegs = 216;
static_assert(128 * kCtrlRegs + 256 * kSoftmaxRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kNumWG = 2;
constexpr int kMaxS = 2;  // smem stages
constexpr int kMaxT = 4;  // TMEM stages
constexpr int kMaxRegChunks = 5;  // rows up to 160 columns are held in registers
constexpr uint32_t kMaxSmem = 232448;     // 227 KB per CTA on sm_100-class parts
constexpr uint32_t kMinSmem = 118 * 1024; // forces one resident CTA per SM

struct Params {
  const int32_t* perm;  // [B, n]; unused when identity
  const float* gate;    // [B, n, Hq] logits or nullptr
  __nv_bfloat16* out;
  int32_t* err;
  int B, n, Hq, Hkv, g, Bt;
  int left, right, span_pad;
  int causal, accumulate, identity;
  float scale_log2;
  int tiles_per_seq, num_tiles;
  int s_stages, t_stages, cols_stage, tmem_alloc;
  int num_wg;  // softmax warpgroups taking alternate tiles (1 or 2)
  uint32_t qk_bytes, stage_bytes, sig_off, bar_off;
  long long rows_q;  // B * n * Hq: bound of the scatter row index
  long long timeout_cycles;
};

// ------------------------------------------------------------------ layout
struct Bars {
  uint32_t base;
  // smem-stage barriers
  __device__ uint32_t full(int s) const { return base + 8u * s; }
  __device__ uint32_t empty(int s) const { return base + 8u * (kMaxS + s); }
  __device__ uint32_t pfull(int s) const { return base + 8u * (2 * kMaxS + s); }
  // TMEM-stage barriers
  __device__ uint32_t sfull(int t) const { return base + 8u * (3 * kMaxS + t); }
  __device__ uint32_t ofull(int t) const { return base + 8u * (3 * kMaxS + kMaxT + t); }
  __device__ uint32_t tempty(int t) const { return base + 8u * (3 * kMaxS + 2 * kMaxT + t); }
  __device__ uint32_t drain() const { return base + 8u * (3 * kMaxS + 3 * kMaxT); }
  static constexpr uint32_t kBytes = 8u * (3 * kMaxS + 3 * kMaxT + 1);
};

struct TileCoord {
  int b, kvh, p0;
};

__device__ __forceinline__ TileCoord decode(const Params& P, int tile) {
  const int seq = tile / P.tiles_per_seq;
  TileCoord c;
  c.b = seq / P.Hkv;
  c.kvh = seq - c.b * P.Hkv;
  c.p0 = (tile - seq * P.tiles_per_seq) * P.Bt;
  return c;
}

// Bounded wait on this kernel's timeout and error word.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Params& P,
                                             volatile int* abort_flag) {
  return bounded_wait(bar, parity, P.timeout_cycles, P.err, abort_flag);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Params& P,
                                          volatile int* abort_flag) {
  const bool ok = wait_bounded(bar, parity, P, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ roles
template <int D>
__device__ void producer_role(const Params& P, const CUtensorMap* tq, const CUtensorMap* tk,
                              const CUtensorMap* tv, uint8_t* smem, uint32_t sbase,
                              const Bars& bars, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  bool issued[kMaxS] = {false, false};
  uint32_t issued_par[kMaxS] = {0, 0};
  int it = 0;
  for (int tile = blockIdx.x; tile < P.num_tiles; tile += gridDim.x, ++it) {
    const int s = it % P.s_stages;
    const uint32_t ph = uint32_t(it / P.s_stages) & 1u;
    if (!warp_wait(bars.empty(s), ph ^ 1u, P, abort_flag)) break;
    const TileCoord tc = decode(P, tile);
    int32_t* sig = reinterpret_cast<int32_t*>(smem + P.sig_off) + s * P.span_pad;
    const int k0 = tc.p0 - P.left;
    const int32_t* perm_b = P.identity ? nullptr : P.perm + size_t(tc.b) * P.n;
    for (int c = lane; c < P.span_pad; c += 32) {
      const int qpos = min(max(k0 + c, 0), P.n - 1);
      int tok = perm_b ? __ldg(perm_b + qpos) : qpos;
      if (unsigned(tok) >= unsigned(P.n)) {
        atomicOr(P.err, SA_ERRBIT_RANGE);
        tok = 0;
      }
      sig[c] = tok;
    }
    __threadfence_block();
    __syncwarp();
    const uint32_t full = bars.full(s);
    if (lane == 0) mbar_arrive_expect_tx(full, uint32_t(kBM + 2 * P.span_pad) * D * 2u);
    __syncwarp();
    const uint32_t q_dst = sbase + uint32_t(s) * P.stage_bytes;
    const uint32_t k_dst = q_dst + kBM * D * 2;
    const uint32_t v_dst = q_dst + P.qk_bytes;
    const int row_base_q = tc.b * P.n;
    {  // Q: 32 groups of four rows, one per lane
      int rows[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = 4 * lane + u;
        const int t = r / P.g;
        const int j = r - t * P.g;
        const int tok = sig[P.left + t];
        rows[u] = (row_base_q + tok) * P.Hq + tc.kvh * P.g + j;
      }
#pragma unroll
      for (int kb = 0; kb < D / 64; ++kb)
        tma_gather4(q_dst + kb * (kBM * 128) + lane * 512, tq, kb * 64, rows[0], rows[1], rows[2],
                    rows[3], full);
    }
    for (int grp = lane; grp < P.span_pad / 4; grp += 32) {  // K and V
      int rows[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) rows[u] = (row_base_q + sig[4 * grp + u]) * P.Hkv + tc.kvh;
#pragma unroll
      for (int kb = 0; kb < D / 64; ++kb) {
        const uint32_t off = kb * (P.span_pad * 128) + grp * 512;
        tma_gather4(k_dst + off, tk, kb * 64, rows[0], rows[1], rows[2], rows[3], full);
        tma_gather4(v_dst + off, tv, kb * 64, rows[0], rows[1], rows[2], rows[3], full);
      }
    }
    issued[s] = true;
    issued_par[s] = ph;
  }
  if (*abort_flag) {  // let this CTA's own copies land before smem is released
    for (int s = 0; s < P.s_stages; ++s)
      if (issued[s]) {
        const long long t0 = clock64();
        while (!mbar_try_wait(bars.full(s), issued_par[s]) && clock64() - t0 < kDrainCycles) {
        }
      }
  }
}

template <int D>
__device__ void mma_role(const Params& P, uint32_t sbase, uint32_t tmem_base, const Bars& bars,
                         volatile int* abort_flag) {
  const int S = P.s_stages, T = P.t_stages;
  const uint32_t q_bytes = kBM * D * 2;
  auto qk = [&](int it) -> bool {
    const int s = it % S, ts = it % T;
    if (!wait_bounded(bars.full(s), uint32_t(it / S) & 1u, P, abort_flag)) return false;
    if (!wait_bounded(bars.tempty(ts), (uint32_t(it / T) & 1u) ^ 1u, P, abort_flag)) return false;
    tc_fence_after();
    const uint32_t d = tmem_base + uint32_t(ts * P.cols_stage);
    const uint32_t qa = sbase + uint32_t(s) * P.stage_bytes;
    const uint32_t ka = qa + q_bytes;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t koff = uint32_t(kk & 3) * 32u;
      const uint64_t a = sdesc_sw128(qa + (kk >> 2) * (kBM * 128) + koff, 16, 1024);
      for (int n0 = 0; n0 < P.span_pad; n0 += 256) {
        const int nn = min(256, P.span_pad - n0);
        const uint64_t bd =
            sdesc_sw128(ka + (kk >> 2) * (P.span_pad * 128) + n0 * 128 + koff, 16, 1024);
        umma_bf16(d + n0, a, bd, idesc_bf16(kBM, nn, 0), kk > 0 ? 1u : 0u);
      }
    }
    umma_commit(bars.sfull(ts));
    return true;
  };
  auto pv = [&](int it) -> bool {
    const int s = it % S, ts = it % T;
    if (!wait_bounded(bars.pfull(s), uint32_t(it / S) & 1u, P, abort_flag)) return false;
    tc_fence_after();
    const uint32_t o = tmem_base + uint32_t(ts * P.cols_stage);
    const uint32_t pa = sbase + uint32_t(s) * P.stage_bytes;
    const uint32_t va = pa + P.qk_bytes;
    const uint32_t idesc = idesc_bf16(kBM, D, 1);
    const int ksteps = P.span_pad / 16;
    for (int kk = 0; kk < ksteps; ++kk) {
      const uint64_t a = sdesc_sw128(pa + (kk >> 2) * (kBM * 128) + (kk & 3) * 32, 16, 1024);
      const uint64_t bd = sdesc_sw128(va + kk * 2048, P.span_pad * 128, 1024);
      umma_bf16(o, a, bd, idesc, kk > 0 ? 1u : 0u);
    }
    umma_commit(bars.ofull(ts));
    umma_commit(bars.empty(s));
    return true;
  };
  const bool overlap = (S >= 2) && (T >= 2);
  bool ok = true;
  int it = 0;
  for (int tile = blockIdx.x; tile < P.num_tiles; tile += gridDim.x, ++it) {
    if (!overlap && it > 0 && !pv(it - 1)) { ok = false; break; }
    if (!qk(it)) { ok = false; break; }
    if (overlap && it > 0 && !pv(it - 1)) { ok = false; break; }
  }
  if (ok && it > 0) pv(it - 1);
  // All MMAs this thread issued complete before TMEM can be released.
  umma_commit(bars.drain());
  const long long t0 = clock64();
  while (!mbar_try_wait(bars.drain(), 0) && clock64() - t0 < kDrainCycles) {
  }
}

// Softmax + epilogue warpgroups.  NCH > 0: the row's NCH*32 columns are read
// from TMEM once and kept in registers; NCH == 0: wider spans, two passes
// over TMEM in 32-column chunks.
template <int D, int NCH, bool kCausal>
__device__ void softmax_role(const Params& P, uint8_t* smem, uint32_t tmem_base, const Bars& bars,
                             volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = (warp - kFirstSoftmaxWarp) >> 2;
  const int quad = warp & 3;  // TMEM lane quadrant this warp may access
  const int r = quad * 32 + lane;
  const int t = r / P.g;
  const int j = r - t * P.g;
  const int S = P.s_stages, T = P.t_stages;
  int it = 0;
  for (int tile = blockIdx.x; tile < P.num_tiles; tile += gridDim.x, ++it) {
    if (wg >= P.num_wg || it % P.num_wg != wg) continue;
    const int s = it % S, ts = it % T;
    const uint32_t ph_s = uint32_t(it / S) & 1u, ph_t = uint32_t(it / T) & 1u;
    const TileCoord tc = decode(P, tile);
    if (!warp_wait(bars.sfull(ts), ph_t, P, abort_flag)) break;
    if (!warp_wait(bars.full(s), ph_s, P, abort_flag)) break;  // sigma smem visibility
    tc_fence_after();
    const int32_t* sig = reinterpret_cast<const int32_t*>(smem + P.sig_off) + s * P.span_pad;
    bool row_valid = tc.p0 + t < P.n;
    RowCtx rc;
    rc.sig_p = sig[P.left + t];
    if (row_valid && unsigned(rc.sig_p) >= unsigned(P.n)) {  // never expected: record and skip
      atomicOr(P.err, SA_ERRBIT_INTERNAL);
      row_valid = false;
    }
    rc.lo = max(t, P.left - tc.p0);
    rc.hi = row_valid ? min(t + P.left + P.right, P.n - 1 - tc.p0 + P.left) : rc.lo - 1;
    rc.wlo = rc.lo;
    rc.whi = rc.hi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      rc.wlo = max(rc.wlo, __shfl_xor_sync(0xffffffffu, rc.wlo, o));
      rc.whi = min(rc.whi, __shfl_xor_sync(0xffffffffu, rc.whi, o));
    }
    rc.scale_log2 = P.scale_log2;
    const uint32_t trow = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(ts * P.cols_stage);
    uint8_t* pbase = smem + size_t(s) * P.stage_bytes;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};

    if constexpr (NCH > 0) {
      uint32_t v[NCH][32];
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) tmem_ld32_async(trow + ch * 32, v[ch]);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) reg_fence(v[ch]);
      float mx = -INFINITY;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) mx = fmaxf(mx, mask_chunk<kCausal>(v[ch], sig, ch * 32, rc));
      const float ms = (mx == -INFINITY) ? 0.f : mx * rc.scale_log2;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        exp_store_chunk(v[ch], ms, rc.scale_log2, pbase, r, ch * 32, acc);
    } else {
      const int nch = P.span_pad / 32;
      float mx = -INFINITY;
      for (int ch = 0; ch < nch; ++ch) {
        uint32_t v[32];
        tmem_ld32(trow + ch * 32, v);
        mx = fmaxf(mx, mask_chunk<kCausal>(v, sig, ch * 32, rc));
      }
      const float ms = (mx == -INFINITY) ? 0.f : mx * rc.scale_log2;
      for (int ch = 0; ch < nch; ++ch) {
        uint32_t v[32];
        tmem_ld32(trow + ch * 32, v);
        mask_chunk<kCausal>(v, sig, ch * 32, rc);
        exp_store_chunk(v, ms, rc.scale_log2, pbase, r, ch * 32, acc);
      }
    }
    const float l = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.pfull(s));

    // epilogue: O / l (* gate, + previous), bf16, row sigma[p0+t] of out
    if (!warp_wait(bars.ofull(ts), ph_t, P, abort_flag)) break;
    tc_fence_after();
    float mul = l > 0.f ? 1.f / l : 0.f;
    const size_t orow =
        row_valid ? (size_t(tc.b) * P.n + rc.sig_p) * P.Hq + size_t(tc.kvh) * P.g + j : 0;
    if (P.gate != nullptr && row_valid) mul *= 1.f / (1.f + expf(-P.gate[orow]));
    __nv_bfloat16* op = P.out + orow * D;
    uint32_t o[D / 32][32];
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) tmem_ld32_async(trow + ch * 32, o[ch]);
    tmem_wait_ld();
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) reg_fence(o[ch]);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.tempty(ts));  // O is in registers: TMEM stage free
    if (row_valid) {
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint4* dst = reinterpret_cast<uint4*>(op + ch * 32);
        uint4 prev[4];
        if (P.accumulate) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) prev[q4] = dst[q4];
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[ch][q4 * 8 + e]) * mul;
          if (P.accumulate) {
            const __nv_bfloat162* pv2 = reinterpret_cast<const __nv_bfloat162*>(&prev[q4]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 pf = __bfloat1622float2(pv2[e]);
              f[2 * e] += pf.x;
              f[2 * e + 1] += pf.y;
            }
          }
          dst[q4] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                               pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
        }
      }
    }
  }
}

template <int D, int NCH>
__device__ __forceinline__ void softmax_dispatch(const Params& P, uint8_t* smem,
                                                 uint32_t tmem_base, const Bars& bars,
                                                 volatile int* abort_flag) {
  if (P.causal)
    softmax_role<D, NCH, true>(P, smem, tmem_base, bars, abort_flag);
  else
    softmax_role<D, NCH, false>(P, smem, tmem_base, bars, abort_flag);
}

template <int D, int NCH>
__global__ void __launch_bounds__(kThreads, 1)
    sa_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ Params P) {
  extern __shared__ uint8_t smem_raw[];
  // Align by pointer arithmetic on the shared array (not through an integer)
  // so the compiler keeps the shared address space: ld/st.shared, not generic.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  Bars bars;
  bars.base = sbase + P.bar_off;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P.bar_off + Bars::kBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.bar_off + Bars::kBytes + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxS; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
      mbar_init(bars.pfull(s), 4);
    }
    for (int t = 0; t < kMaxT; ++t) {
      mbar_init(bars.sfull(t), 1);
      mbar_init(bars.ofull(t), 1);
      mbar_init(bars.tempty(t), 4);
    }
    mbar_init(bars.drain(), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kTmemWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(uint32_t(P.tmem_alloc))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Each branch ends with the CTA-wide barrier of its own so that no code
  // runs after the branches under two register limits.
  if (warp >= kFirstSoftmaxWarp) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    softmax_dispatch<D, NCH>(P, smem, tmem_base, bars, abort_flag);
    tc_fence_before();
    __syncthreads();
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    if (warp == kProducerWarp) {
      producer_role<D>(P, &tm_q, &tm_k, &tm_v, smem, sbase, bars, abort_flag);
    } else if (warp == kMmaWarp) {
      if ((threadIdx.x & 31) == 0) mma_role<D>(P, sbase, tmem_base, bars, abort_flag);
      __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTmemWarp) {
      tc_fence_after();
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(uint32_t(P.tmem_alloc))
                   : "memory");
    }
  }
}

// ------------------------------------------------------------------ host
struct Config {
  int Bt, left, right, span_pad, s_stages, t_stages, cols_stage, tmem_alloc, num_wg;
  uint32_t qk_bytes, stage_bytes, sig_off, bar_off, smem_bytes;
};

static uint32_t round_up(uint32_t x, uint32_t m) { return (x + m - 1) / m * m; }

static bool device_has_tcgen05(int* sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (sm_count) cudaDeviceGetAttribute(sm_count, cudaDevAttrMultiProcessorCount, dev);
  // This library is built for sm_103a only.
  return major == 10 && minor == 3;
}

static bool make_config(const Problem& pb, Path path, Config& c) {
  if (pb.d != 64 && pb.d != 128) return false;
  if (kBM % pb.g != 0) return false;
  c.Bt = kBM / pb.g;
  if (path == kPathSA) {
    c.left = c.right = pb.window / 2;
  } else {
    c.left = pb.window_swa - 1;
    c.right = 0;
  }
  const long long span = (long long)c.Bt + c.left + c.right;
  if (span > 512) return false;
  c.span_pad = int(round_up(uint32_t(span), 32));
  c.cols_stage = c.span_pad > pb.d ? c.span_pad : pb.d;
  if (c.cols_stage > 512) return false;
  c.t_stages = 512 / c.cols_stage;
  if (c.t_stages > kMaxT) c.t_stages = kMaxT;
  uint32_t alloc = 32;
  while (alloc < uint32_t(c.t_stages * c.cols_stage)) alloc <<= 1;
  c.tmem_alloc = int(alloc);
  const uint32_t q_bytes = kBM * pb.d * 2;
  const uint32_t k_bytes = uint32_t(c.span_pad) * pb.d * 2;
  const uint32_t p_bytes = kBM * round_up(uint32_t(c.span_pad), 64) * 2;
  c.qk_bytes = round_up(q_bytes + k_bytes > p_bytes ? q_bytes + k_bytes : p_bytes, 1024);
  const uint32_t v_bytes = round_up(k_bytes, 1024);
  c.stage_bytes = c.qk_bytes + v_bytes;
  for (int s = kMaxS; s >= 1; --s) {
    const uint32_t sig_off = uint32_t(s) * c.stage_bytes;
    const uint32_t bar_off = round_up(sig_off + uint32_t(s) * c.span_pad * 4, 64);
    const uint32_t total = bar_off + Bars::kBytes + 16 + 1024;  // + slot, flag, alignment slack
    if (total <= kMaxSmem) {
      c.s_stages = s;
      c.sig_off = sig_off;
      c.bar_off = bar_off;
      c.smem_bytes = total < kMinSmem ? kMinSmem : total;
      // Tile `it` goes to warpgroup it % num_wg, smem stage it % S and TMEM
      // stage it % T.  Each warpgroup must see every phase of the barriers
      // it waits on, in order (a parity wait cannot tell phase k from k+2),
      // so two warpgroups need S and T both multiples of 2.
      c.num_wg = (c.s_stages >= 2 && c.t_stages >= 2) ? kNumWG : 1;
      if (c.num_wg == 2) c.t_stages &= ~1;
      return true;
    }
  }
  return false;
}

// Row-gather view of a BSHD bf16 tensor: [rows, d] with 64-element boxes of
// one row, 128-byte swizzle.
static bool make_row_map(CUtensorMap* m, const void* base, uint64_t rows, int d) {
  return encode_row_map(m, base, rows, d, 1);
}

template <int D, int NCH>
static cudaError_t launch_one(int grid, uint32_t smem, cudaStream_t stream, const CUtensorMap& mq,
                              const CUtensorMap& mk, const CUtensorMap& mv, const Params& P) {
  cudaError_t ce = cudaFuncSetAttribute(sa_tc_kernel<D, NCH>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (ce != cudaSuccess) return ce;
  cudaFuncAttributes fa;
  ce = cudaFuncGetAttributes(&fa, sa_tc_kernel<D, NCH>);
  if (ce != cudaSuccess) return ce;
  // The register split assumes the launch allocation; never launch otherwise.
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  int resident = 0;  // a CTA of this variant must fit on an SM (registers and smem)
  ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, sa_tc_kernel<D, NCH>, kThreads,
                                                     smem);
  if (ce != cudaSuccess) return ce;
  if (resident < 1) return cudaErrorInvalidConfiguration;
  sa_tc_kernel<D, NCH><<<grid, kThreads, smem, stream>>>(mq, mk, mv, P);
  return cudaGetLastError();
}

// NCH = span_pad / 32 when the whole row fits in registers, else 0.
template <int D>
static cudaError_t launch_variant(int nch, int grid, uint32_t smem, cudaStream_t stream,
                                  const CUtensorMap& mq, const CUtensorMap& mk,
                                  const CUtensorMap& mv, const Params& P) {
  switch (nch) {
    case 1: return launch_one<D, 1>(grid, smem, stream, mq, mk, mv, P);
    case 2: return launch_one<D, 2>(grid, smem, stream, mq, mk, mv, P);
    case 3: return launch_one<D, 3>(grid, smem, stream, mq, mk, mv, P);
    case 4: return launch_one<D, 4>(grid, smem, stream, mq, mk, mv, P);
    case 5: return launch_one<D, 5>(grid, smem, stream, mq, mk, mv, P);
    default: return launch_one<D, 0>(grid, smem, stream, mq, mk, mv, P);
  }
}

}  // namespace tc

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode_row_map(CUtensorMap* m, const void* base, uint64_t rows, int d, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cuuint64_t(d), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(d) * 2};
  const cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace tc {
// Whether the variant was compiled to the launch register count its
// register split assumes (checked once per variant).
template <int D>
static bool regs_ok(int nch) {
  static int cache[6] = {-1, -1, -1, -1, -1, -1};
  const int i = nch < 0 ? 0 : (nch > 5 ? 0 : nch);
  if (cache[i] < 0) {
    cudaFuncAttributes fa;
    cudaError_t ce;
    switch (i) {
      case 1: ce = cudaFuncGetAttributes(&fa, sa_tc_kernel<D, 1>); break;
      case 2: ce = cudaFuncGetAttributes(&fa, sa_tc_kernel<D, 2>); break;
      case 3: ce = cudaFuncGetAttributes(&fa, sa_tc_kernel<D, 3>); break;
      case 4: ce = cudaFuncGetAttributes(&fa, sa_tc_kernel<D, 4>); break;
      case 5: ce = cudaFuncGetAttributes(&fa, sa_tc_kernel<D, 5>); break;
      default: ce = cudaFuncGetAttributes(&fa, sa_tc_kernel<D, 0>); break;
    }
    cache[i] = (ce == cudaSuccess && fa.numRegs == kLaunchRegs) ? 1 : 0;
  }
  return cache[i] == 1;
}
}  // namespace tc

bool tc_supported(const Problem& pb, Path path) {
  if (path != kPathSA && path != kPathSWA) return false;
  if (!tc::device_has_tcgen05(nullptr)) return false;
  tc::Config c;
  if (!tc::make_config(pb, path, c)) return false;
  const int nch = c.span_pad / 32 <= tc::kMaxRegChunks ? c.span_pad / 32 : 0;
  return pb.d == 128 ? tc::regs_ok<128>(nch) : tc::regs_ok<64>(nch);
}

sa_status_t launch_tc(const Problem& pb, Path path, const float* gate, int accumulate,
                      cudaStream_t stream) {
  using namespace tc;
  int sms = 0;
  if (!device_has_tcgen05(&sms)) return fail(SA_ERR_UNSUPPORTED, "device is not sm_103");
  Config c;
  if (!make_config(pb, path, c)) return fail(SA_ERR_UNSUPPORTED, "shape does not fit the tcgen05 kernel");
  CUtensorMap mq, mk, mv;
  const uint64_t rows_q = uint64_t(pb.B) * pb.n * pb.Hq;
  const uint64_t rows_kv = uint64_t(pb.B) * pb.n * pb.Hkv;
  if (!make_row_map(&mq, pb.q, rows_q, pb.d) || !make_row_map(&mk, pb.k, rows_kv, pb.d) ||
      !make_row_map(&mv, pb.v, rows_kv, pb.d))
    return fail(SA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  Params P;
  std::memset(&P, 0, sizeof(P));
  P.perm = pb.perm;
  P.gate = gate;
  P.out = static_cast<__nv_bfloat16*>(pb.out);
  P.err = pb.err;
  P.B = pb.B;
  P.n = pb.n;
  P.Hq = pb.Hq;
  P.Hkv = pb.Hkv;
  P.g = pb.g;
  P.Bt = c.Bt;
  P.left = c.left;
  P.right = c.right;
  P.span_pad = c.span_pad;
  P.causal = (path == kPathSA) ? pb.causal : 0;
  P.accumulate = accumulate;
  P.identity = (path == kPathSWA) ? 1 : 0;
  P.scale_log2 = pb.scale * 1.4426950408889634f;
  P.tiles_per_seq = (pb.n + c.Bt - 1) / c.Bt;
  P.num_tiles = P.tiles_per_seq * pb.B * pb.Hkv;
  P.s_stages = c.s_stages;
  P.t_stages = c.t_stages;
  P.cols_stage = c.cols_stage;
  P.tmem_alloc = c.tmem_alloc;
  P.num_wg = c.num_wg;
  P.rows_q = (long long)pb.B * pb.n * pb.Hq;
  P.qk_bytes = c.qk_bytes;
  P.stage_bytes = c.stage_bytes;
  P.sig_off = c.sig_off;
  P.bar_off = c.bar_off;
  P.timeout_cycles = wait_limit_cycles();
  const int grid = P.num_tiles < sms ? P.num_tiles : sms;
  const int nch = c.span_pad / 32 <= kMaxRegChunks ? c.span_pad / 32 : 0;
  cudaError_t ce;
  if (pb.d == 128)
    ce = launch_variant<128>(nch, grid, c.smem_bytes, stream, mq, mk, mv, P);
  else
    ce = launch_variant<64>(nch, grid, c.smem_bytes, stream, mq, mk, mv, P);
  if (ce == cudaSuccess) ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "tcgen05 kernel launch: %s", cudaGetErrorString(ce));
  return SA_OK;
}

}  // namespace sa
