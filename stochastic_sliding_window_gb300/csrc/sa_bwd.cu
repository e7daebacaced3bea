// tcgen05 backward pass of SA / SWA and of the gated merge: gradients with
// respect to Q, K, V and the gate logits.
//
// The Stochastic Attention summary uses the gated SA + SWA pair to pretrain
// a model from scratch ("Main contributions", item 3), which needs these
// gradients; the pages print no formula, so they follow from the forward
// definition ("Core mechanism" steps 1-3, the causal rule of "Theoretical
// properties", the "Gated SA and SWA" equation) by the chain rule.  With
// p = softmax(scale q k^T) over a row's window, upstream gradient u = g * dy
// (g = sigmoid of the row's gate logit, 1 without a gate):
//   dP = dy V^T,   D = sum_j p dP (= <dy, y>),   dS = g p (dP - D)
//   dQ = scale dS K,   dK = scale dS^T Q,   dV = (g p)^T dy,
//   d(gate logit) = g (1 - g) D.
// Everything runs in the permuted order, over the same tiles as the forward
// kernels: a tile is Bt = 128/g consecutive permuted positions of one
// (sequence, kv head) pair stacked with the g query heads (128 MMA rows).
//
// Two kernels, both one 256-thread CTA per SM walking tiles; the two warps
// of a TMEM lane quarter share its 32 rows (one MMA row per lane) and split
// each row's 32-column pieces:
//   sa_bwd_dq_kernel   query tiles: gathers the tile's Q and dY rows and the
//                      K and V rows of its key span into shared memory (the
//                      next tile's rows while this one is computed);
//                      S = Q K^T and dP = dY V^T into TMEM; per row the
//                      log-sum-exp and D from its whole window, then
//                      dS (bf16) over S; dQ = dS K; dQ rows scattered to
//                      sigma[p].  Writes each row's log-sum-exp and D for the
//                      second kernel, and the gate-logit gradient.
//   sa_bwd_dkv_kernel  key tiles of 128 permuted positions: K and V rows in
//                      shared memory; the query positions whose window
//                      covers a key of the tile are walked in chunks of 128
//                      rows: S^T = K Q^T and dP^T = V dY^T into TMEM, then
//                      P^T and dS^T (bf16, from the stored log-sum-exp and D)
//                      over them; dV += P^T dY and dK += dS^T Q accumulate in
//                      TMEM across the chunks; each key's complete dK, dV
//                      rows are written once.  No atomics anywhere.
// Results go to bf16 outputs, or to fp32 buffers (stored, or added for the
// second path of the gated merge) that a conversion kernel turns into bf16.
// Every wait is bounded (SA_ERRBIT_TIMEOUT); MMAs and copies in flight are
// drained before tensor and shared memory are released.
#include "sa_internal.h"
#include "sa_tc_common.cuh"

#include <cstring>

namespace sa {
namespace bwd {

using namespace tcc;

constexpr int kThreads = 256;
constexpr uint32_t kMaxSmem = 232448;
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* dy;
  const int32_t* perm;  // [B, n]; nullptr: identity (SWA)
  const float* gate;    // [B, n, Hq] logits or nullptr
  float* lse2;          // [B, n, Hq] log2 of (row normaliser / gate), written by dq
  float* dsum;          // [B, n, Hq] D of the row, written by dq
  float* dgate;         // [B, n, Hq] gate-logit gradient, or nullptr
  void* dq;             // [B, n, Hq, d]
  void* dk;             // [B, n, Hkv, d]
  void* dv;
  int out_mode;         // 0: bf16 store, 1: fp32 store, 2: fp32 add
  int32_t* err;
  int B, n, Hq, Hkv, g, log2g, Bt;
  int left, right;      // window: keys at permuted positions [p - left, p + right]
  int span_pad;         // dq: key span of a query tile, rounded up to 32
  int causal;
  float scale, scale_log2;
  int num_tiles, tiles_per_seq;
  int tmem_alloc;
  uint32_t off_q, off_dy, off_k, off_v, off_sig, off_col, off_bar;
  long long timeout_cycles;
};

// Barrier slots after off_bar: the MMA barrier, the exit drain barrier, then
// the TMEM address slot and the abort flag.
enum : uint32_t { kBarMma = 0, kBarDrain = 1, kNumBars = 2 };

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// A from TMEM, B from shared memory, D in TMEM.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// cp.async of `rows` rows of D bf16 (given by row_of(i) as an element
// offset) into the 128-byte-swizzled K-major layout with K-blocks
// `kb_stride` bytes apart, spread over the CTA's threads.
template <int D, class RowFn>
__device__ __forceinline__ void gather_rows(uint32_t dst, uint32_t kb_stride, int rows,
                                            const __nv_bfloat16* base, RowFn row_of) {
  constexpr int CPR = D / 8;
  for (int idx = threadIdx.x; idx < rows * CPR; idx += kThreads) {
    const int r = idx / CPR, c = idx - (idx / CPR) * CPR;
    const int kb = c >> 3, c8 = c & 7;
    cp_async16(dst + kb * kb_stride + r * 128 + ((c8 ^ (r & 7)) << 4), base + row_of(r) + c * 8);
  }
}

// All threads agree on a bounded wait of the MMA barrier (false: give up).
__device__ __forceinline__ bool cta_wait(uint32_t bar, uint32_t parity, const Params& P,
                                         volatile int* abort_flag) {
  const bool ok = bounded_wait(bar, parity, P.timeout_cycles, P.err, abort_flag);
  return !__syncthreads_or(ok ? 0 : 1);
}

// Common CTA set-up: barriers, flag, TMEM.  Returns the TMEM base address.
__device__ __forceinline__ uint32_t cta_setup(const Params& P, uint8_t* smem, uint32_t bars,
                                              volatile int*& abort_flag) {
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P.off_bar + 8 * kNumBars);
  abort_flag = reinterpret_cast<volatile int*>(smem + P.off_bar + 8 * kNumBars + 4);
  if (threadIdx.x == 0) {
    mbar_init(bars + 8 * kBarMma, 1);
    mbar_init(bars + 8 * kBarDrain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(uint32_t(P.tmem_alloc))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return *tmem_slot;
}

// Common exit: MMAs this CTA issued complete, then TMEM is released.
__device__ __forceinline__ void cta_teardown(const Params& P, uint32_t bars, uint32_t tmem_base) {
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (threadIdx.x == 0) {
    umma_commit(bars + 8 * kBarDrain);
    const long long t0 = clock64();
    while (!mbar_try_wait(bars + 8 * kBarDrain, 0) && clock64() - t0 < kDrainCycles) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(uint32_t(P.tmem_alloc))
                 : "memory");
  }
}

// One output row of D values (fp32 in registers, `mul` applied) to a bf16
// or fp32 destination row.
template <int D>
__device__ __forceinline__ void write_row(const Params& P, void* base, size_t row,
                                          const uint32_t (&v)[32], int col0, float mul) {
  if (P.out_mode == 0) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + row * D + col0);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
      dst[q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
  } else {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + row * D + col0);
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4) {
      float4 f = make_float4(__uint_as_float(v[4 * q4]) * mul, __uint_as_float(v[4 * q4 + 1]) * mul,
                             __uint_as_float(v[4 * q4 + 2]) * mul,
                             __uint_as_float(v[4 * q4 + 3]) * mul);
      if (P.out_mode == 2) {
        const float4 o = dst[q4];
        f.x += o.x;
        f.y += o.y;
        f.z += o.z;
        f.w += o.w;
      }
      dst[q4] = f;
    }
  }
}

// ------------------------------------------------------------------ dQ
// 256 threads: warp w reads TMEM lane quarter w % 4 (rows 32 (w % 4) ..),
// and the two warps of a quarter split each row's 32-column pieces between
// them (piece ch goes to half ch % 2); row reductions meet in shared memory.
template <int D, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1) sa_bwd_dq_kernel(const __grid_constant__ Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + P.off_bar;
  volatile int* abort_flag;
  const uint32_t tmem_base = cta_setup(P, smem, bars, abort_flag);
  // span column -> token (-1: none), two buffers: this tile's and the next one's
  int32_t* sigbuf = reinterpret_cast<int32_t*>(smem + P.off_sig);
  float* red = reinterpret_cast<float*>(smem + P.off_col);       // [3][2][128] row partials
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, part = warp >> 2;
  const int r = quarter * 32 + lane;  // this thread's TMEM lane = MMA row
  const int t = r >> P.log2g, j = r & (P.g - 1);
  const uint32_t trow = tmem_base + (uint32_t(quarter * 32) << 16);
  const uint32_t sq = sbase + P.off_q, sdy = sbase + P.off_dy, sk = sbase + P.off_k,
                 sv = sbase + P.off_v;
  const int sp = P.span_pad;
  uint32_t mma_phase = 0;
  struct TileAt {
    int p0, kvh;
    size_t tokb, qh;
  };
  auto tile_at = [&](int tile_) {
    const int seq = tile_ / P.tiles_per_seq;
    const int b = seq / P.Hkv;
    TileAt c;
    c.p0 = (tile_ - seq * P.tiles_per_seq) * P.Bt;
    c.kvh = seq - b * P.Hkv;
    c.tokb = size_t(b) * P.n;
    c.qh = size_t(c.kvh) * P.g;
    return c;
  };
  // the tile's span tokens into sg (the caller synchronises before use)
  auto fill_sig = [&](const TileAt& c, int32_t* sg) {
    for (int i = tid; i < sp; i += kThreads) {
      const int pos = c.p0 - P.left + i;
      int tok = -1;
      if (pos >= 0 && pos < P.n) {
        tok = P.perm ? __ldg(P.perm + c.tokb + pos) : pos;
        if (unsigned(tok) >= unsigned(P.n)) {
          atomicOr(P.err, SA_ERRBIT_RANGE);
          tok = -1;
        }
      }
      sg[i] = tok;
    }
  };
  // Q and dY rows of the tile (r = t*g + j), K or V rows of the span; rows
  // past the sequence end read token 0 and are never written.
  auto gather_qdy = [&](const TileAt& c, const int32_t* sg) {
    auto qrow = [&](int rr) {
      const int tk = max(sg[P.left + (rr >> P.log2g)], 0);
      return ((c.tokb + tk) * P.Hq + c.qh + (rr & (P.g - 1))) * D;
    };
    gather_rows<D>(sq, kBM * 128, kBM, P.q, qrow);
    gather_rows<D>(sdy, kBM * 128, kBM, P.dy, qrow);
  };
  auto gather_kv = [&](const TileAt& c, const int32_t* sg, uint32_t dst,
                       const __nv_bfloat16* src) {
    auto krow = [&](int s_) { return ((c.tokb + max(sg[s_], 0)) * P.Hkv + c.kvh) * D; };
    gather_rows<D>(dst, sp * 128, sp, src, krow);
  };
  // The operands of the first tile; every later tile's are gathered while
  // the tile before it is computed: its Q, dY and V rows once that tile's
  // S and dP MMAs are done, its K rows once that tile's dQ MMA is.
  int cur = 0;
  if (int(blockIdx.x) < P.num_tiles) {
    const TileAt c0 = tile_at(blockIdx.x);
    fill_sig(c0, sigbuf);
    __syncthreads();
    gather_qdy(c0, sigbuf);
    gather_kv(c0, sigbuf, sk, P.k);
    gather_kv(c0, sigbuf, sv, P.v);
  }
  for (int tile = blockIdx.x; tile < P.num_tiles; tile += gridDim.x, cur ^= 1) {
    const TileAt c = tile_at(tile);
    const int p0 = c.p0;
    const size_t tokb = c.tokb, qh = c.qh;
    const int32_t* sig = sigbuf + cur * sp;
    int32_t* sig_nx = sigbuf + (cur ^ 1) * sp;
    const int next = tile + int(gridDim.x);
    const bool has_next = next < P.num_tiles;
    asm volatile("cp.async.wait_all;" ::: "memory");
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16(kBM, sp, 0);
      const uint64_t a0 = sdesc_sw128(sq, 16, 1024), y0 = sdesc_sw128(sdy, 16, 1024);
      const uint64_t b0 = sdesc_sw128(sk, 16, 1024), v0 = sdesc_sw128(sv, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t da = uint64_t((kk >> 2) * (kBM * 128 / 16) + (kk & 3) * 2);
        const uint64_t db = uint64_t((kk >> 2) * (sp * 128 / 16) + (kk & 3) * 2);
        umma_bf16(tmem_base, a0 + da, b0 + db, id, kk > 0 ? 1u : 0u);           // S
        umma_bf16(tmem_base + sp, y0 + da, v0 + db, id, kk > 0 ? 1u : 0u);      // dP
      }
      umma_commit(bars + 8 * kBarMma);
    }
    if (has_next) fill_sig(tile_at(next), sig_nx);  // overlaps the MMAs
    if (!cta_wait(bars + 8 * kBarMma, mma_phase, P, abort_flag)) break;
    mma_phase ^= 1;
    tc_fence_after();
    // Q, dY and V are free: the next tile's rows land during the passes
    // (cta_wait above also ordered sig_nx's writes before these reads)
    TileAt cn{};
    if (has_next) {
      cn = tile_at(next);
      gather_qdy(cn, sig_nx);
      gather_kv(cn, sig_nx, sv, P.v);
    }

    // Per row: window band in span columns, its token, gate.
    const int sig_p = sig[P.left + t];
    const bool row_valid = sig_p >= 0;
    const int lo = max(t, P.left - p0);
    const int hi = row_valid ? min(t + P.left + P.right, P.n - 1 - p0 + P.left) : -1;
    const size_t orow = (tokb + max(sig_p, 0)) * P.Hq + qh + j;
    auto bits_of = [&](int ch) {
      uint32_t bits = band_bits(lo, hi, ch * 32);
      if (kCausal && bits) {
        const int4* s4p = reinterpret_cast<const int4*>(sig + ch * 32);
        uint32_t cw = 0;
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const int4 s4 = s4p[e4];
          cw |= (s4.x <= sig_p ? 1u : 0u) << (4 * e4);
          cw |= (s4.y <= sig_p ? 1u : 0u) << (4 * e4 + 1);
          cw |= (s4.z <= sig_p ? 1u : 0u) << (4 * e4 + 2);
          cw |= (s4.w <= sig_p ? 1u : 0u) << (4 * e4 + 3);
        }
        bits &= cw;
      }
      return bits;
    };
    const int nch = sp / 32;
    // This row's words of its pieces ch = part + 2k (k < 4: spans of up to
    // 256 keys), built once for the three passes; picked by a select chain
    // (an indexed register array would live in local memory).
    uint32_t wb0 = 0u, wb1 = 0u, wb2 = 0u, wb3 = 0u;
    if (part < nch) wb0 = bits_of(part);
    if (part + 2 < nch) wb1 = bits_of(part + 2);
    if (part + 4 < nch) wb2 = bits_of(part + 4);
    if (part + 6 < nch) wb3 = bits_of(part + 6);
    auto word = [&](int ch) {
      const int k = (ch - part) >> 1;
      return k == 0 ? wb0 : (k == 1 ? wb1 : (k == 2 ? wb2 : wb3));
    };
    // pass 1: the attended maximum of the raw scores (this half's pieces)
    float mx = -INFINITY;
#pragma unroll 1
    for (int ch = part; ch < nch; ch += 2) {
      uint32_t s_[32];
      tmem_ld32(trow + ch * 32, s_);
      const uint32_t bits = word(ch);
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if ((bits >> e) & 1u) mx = fmaxf(mx, __uint_as_float(s_[e]));
    }
    red[part * kBM + r] = mx;
    __syncthreads();
    mx = fmaxf(red[r], red[kBM + r]);
    const float ms = mx == -INFINITY ? 0.f : mx * P.scale_log2;
    // pass 2: normaliser l and sum of e * dP
    float l = 0.f, pd = 0.f;
#pragma unroll 1
    for (int ch = part; ch < nch; ch += 2) {
      uint32_t s_[32], dp[32];
      tmem_ld32(trow + ch * 32, s_);
      tmem_ld32(trow + sp + ch * 32, dp);
      const uint32_t bits = word(ch);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float ex = (bits >> e) & 1u ? fast_exp2(fmaf(__uint_as_float(s_[e]), P.scale_log2, -ms))
                                          : 0.f;
        l += ex;
        pd = fmaf(ex, __uint_as_float(dp[e]), pd);
      }
    }
    red[2 * kBM + part * kBM + r] = l;
    red[4 * kBM + part * kBM + r] = pd;
    __syncthreads();
    l = red[2 * kBM + r] + red[3 * kBM + r];
    pd = red[4 * kBM + r] + red[5 * kBM + r];
    const float dsum = l > 0.f ? pd / l : 0.f;
    float gl = 1.f;
    if (P.gate != nullptr && row_valid) gl = 1.f / (1.f + expf(-P.gate[orow]));
    // p' = g * p = 2^(s * scale * log2e - lse2'), lse2' = log2(l) + ms - log2(g)
    const float lse2 = ms + log2f(l > 0.f ? l : 1.f) - log2f(gl);
    if (row_valid && part == 0) {
      P.lse2[orow] = lse2;
      P.dsum[orow] = dsum;
      if (P.dgate != nullptr) P.dgate[orow] = gl * (1.f - gl) * dsum;
    }
    // pass 3: dS = p' (dP - D), bf16, over the first 16 columns of the same
    // 32-column S piece (the two warps of a row work on different pieces at
    // once, so nothing may land on a piece the other warp still reads)
#pragma unroll 1
    for (int ch = part; ch < nch; ch += 2) {
      uint32_t s_[32], dp[32];
      tmem_ld32(trow + ch * 32, s_);
      tmem_ld32(trow + sp + ch * 32, dp);
      const uint32_t bits = word(ch);
      uint32_t pk[16];
#pragma unroll
      for (int e2 = 0; e2 < 16; ++e2) {
        float d2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int e = 2 * e2 + u;
          const float p = (bits >> e) & 1u
                              ? fast_exp2(fmaf(__uint_as_float(s_[e]), P.scale_log2, -lse2))
                              : 0.f;
          d2[u] = p * (__uint_as_float(dp[e]) - dsum);
        }
        pk[e2] = pack_bf16x2(d2[0], d2[1]);
      }
      tmem_st16(trow + ch * 32, pk);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    // dQ = dS K: A = dS from TMEM (16 key columns per K step, packed in the
    // first half of each 32-column piece), B = the span's K rows (MN-major)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16(kBM, D, 1);
      uint64_t bd = sdesc_sw128(sk, sp * 128, 1024);
      for (int kk = 0; kk < sp / 16; ++kk) {
        umma_bf16_ts(tmem_base + sp, tmem_base + (kk >> 1) * 32 + (kk & 1) * 8, bd, id,
                     kk > 0 ? 1u : 0u);
        bd += 128;  // 16 key rows of 128 B
      }
      umma_commit(bars + 8 * kBarMma);
    }
    if (!cta_wait(bars + 8 * kBarMma, mma_phase, P, abort_flag)) break;
    mma_phase ^= 1;
    tc_fence_after();
    if (has_next) gather_kv(cn, sig_nx, sk, P.k);  // K is free once dQ = dS K is done
    // tcgen05.ld is warp-collective: every lane loads, valid rows store.
#pragma unroll 1
    for (int ch = part; ch < D / 32; ch += 2) {
      uint32_t o[32];
      tmem_ld32(trow + sp + ch * 32, o);
      if (row_valid) write_row<D>(P, P.dq, orow, o, ch * 32, P.scale);
    }
    tc_fence_before();
    __syncthreads();  // TMEM and this tile's span tokens are reused
  }
  cta_teardown(P, bars, tmem_base);
}

// ------------------------------------------------------------------ dK, dV
// 256 threads as in the dQ kernel (two warps per TMEM lane quarter, pieces
// split between them).  The query chunks' Q and dY rows are double-buffered:
// chunk c + 1 is gathered while chunk c is computed.
template <int D, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1) sa_bwd_dkv_kernel(const __grid_constant__ Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + P.off_bar;
  volatile int* abort_flag;
  const uint32_t tmem_base = cta_setup(P, smem, bars, abort_flag);
  int32_t* ktok = reinterpret_cast<int32_t*>(smem + P.off_sig);  // [128] key tokens (-1: none)
  int32_t* qtok = ktok + kBM;                                    // [2][128] chunk query tokens
  float* col_lse = reinterpret_cast<float*>(smem + P.off_col);   // [2][128] per chunk row
  float* col_d = col_lse + 2 * kBM;                              // [2][128]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, part = warp >> 2;
  const int m = quarter * 32 + lane;  // this thread's key row (TMEM lane)
  const uint32_t trow = tmem_base + (uint32_t(quarter * 32) << 16);
  const uint32_t sk = sbase + P.off_k, sv = sbase + P.off_v;
  const uint32_t chunk_bytes = kBM * D * 2;
  const uint32_t c_st = 0, c_dpt = kBM, c_dv = 2 * kBM, c_dk = 2 * kBM + D;  // TMEM columns
  uint32_t mma_phase = 0;
  for (int tile = blockIdx.x; tile < P.num_tiles; tile += gridDim.x) {
    const int seq = tile / P.tiles_per_seq;
    const int k0 = (tile - seq * P.tiles_per_seq) * kBM;
    const int b = seq / P.Hkv, kvh = seq - (seq / P.Hkv) * P.Hkv;
    const size_t tokb = size_t(b) * P.n;
    if (tid < kBM) {
      const int pos = k0 + tid;
      int tok = -1;
      if (pos < P.n) {
        tok = P.perm ? __ldg(P.perm + tokb + pos) : pos;
        if (unsigned(tok) >= unsigned(P.n)) {
          atomicOr(P.err, SA_ERRBIT_RANGE);
          tok = -1;
        }
      }
      ktok[tid] = tok;
    }
    __syncthreads();
    auto krow = [&](int mm) { return ((tokb + max(ktok[mm], 0)) * P.Hkv + kvh) * D; };
    gather_rows<D>(sk, kBM * 128, kBM, P.k, krow);
    gather_rows<D>(sv, kBM * 128, kBM, P.v, krow);
    // Query positions whose window covers a key of the tile.
    const int qlo = max(0, k0 - P.right);
    const int qhi = min(P.n - 1, k0 + kBM - 1 + P.left);
    const int nchunks = (qhi - qlo + P.Bt) / P.Bt;
    const int kpos = k0 + m;
    const int sig_k = ktok[m];
    const size_t qh = size_t(kvh) * P.g;
    // Tokens, rows and per-row values of chunk c into stage st (every
    // thread; ends with the chunk's copies committed as one group).
    auto prepare = [&](int c, int st) {
      const int c0 = qlo + c * P.Bt;
      int32_t* qt = qtok + st * kBM;
      for (int i = tid; i < P.Bt; i += kThreads) {
        const int pos = c0 + i;
        int tok = -1;
        if (pos <= qhi) {
          tok = P.perm ? __ldg(P.perm + tokb + pos) : pos;
          if (unsigned(tok) >= unsigned(P.n)) tok = -1;  // reported by the dQ kernel
        }
        qt[i] = tok;
      }
      __syncthreads();
      auto qrow = [&](int rr) {
        const int tk = max(qt[rr >> P.log2g], 0);
        return ((tokb + tk) * P.Hq + qh + (rr & (P.g - 1))) * D;
      };
      gather_rows<D>(sbase + P.off_q + st * chunk_bytes, kBM * 128, kBM, P.q, qrow);
      gather_rows<D>(sbase + P.off_dy + st * chunk_bytes, kBM * 128, kBM, P.dy, qrow);
      asm volatile("cp.async.commit_group;" ::: "memory");
      if (tid < kBM) {
        const int tk = qt[tid >> P.log2g];
        const size_t orow = (tokb + max(tk, 0)) * P.Hq + qh + (tid & (P.g - 1));
        col_lse[st * kBM + tid] = tk >= 0 ? P.lse2[orow] : INFINITY;  // 2^(-inf): nothing
        col_d[st * kBM + tid] = tk >= 0 ? P.dsum[orow] : 0.f;
      }
    };
    prepare(0, 0);
    bool alive = true;
    for (int c = 0; c < nchunks && alive; ++c) {
      const int st = c & 1;
      const int c0 = qlo + c * P.Bt;
      asm volatile("cp.async.wait_all;" ::: "memory");  // chunk c (and the tile's K, V)
      fence_proxy_async_smem();
      __syncthreads();
      // The other stage was last read by chunk c - 1, whose MMAs are done.
      if (c + 1 < nchunks) prepare(c + 1, st ^ 1);
      const uint32_t sq = sbase + P.off_q + st * chunk_bytes;
      const uint32_t sdy = sbase + P.off_dy + st * chunk_bytes;
      const int32_t* qt = qtok + st * kBM;
      const float* cl = col_lse + st * kBM;
      const float* cd = col_d + st * kBM;
      if (tid == 0) {
        tc_fence_after();
        const uint32_t id = idesc_bf16(kBM, kBM, 0);
        const uint64_t k0d = sdesc_sw128(sk, 16, 1024), v0d = sdesc_sw128(sv, 16, 1024);
        const uint64_t q0d = sdesc_sw128(sq, 16, 1024), y0d = sdesc_sw128(sdy, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t dd = uint64_t((kk >> 2) * (kBM * 128 / 16) + (kk & 3) * 2);
          umma_bf16(tmem_base + c_st, k0d + dd, q0d + dd, id, kk > 0 ? 1u : 0u);   // S^T
          umma_bf16(tmem_base + c_dpt, v0d + dd, y0d + dd, id, kk > 0 ? 1u : 0u);  // dP^T
        }
        umma_commit(bars + 8 * kBarMma);
      }
      if (!cta_wait(bars + 8 * kBarMma, mma_phase, P, abort_flag)) {
        alive = false;
        break;
      }
      mma_phase ^= 1;
      tc_fence_after();
      // P'^T = 2^(s * scale * log2e - lse2') and dS^T = P'^T (dP^T - D) for
      // attended (key, query row) pairs, bf16 over the first 16 columns of
      // their own 32-column pieces of S^T and dP^T.
#pragma unroll 1
      for (int ch = part; ch < kBM / 32; ch += 2) {
        uint32_t s_[32], dp[32];
        tmem_ld32(trow + c_st + ch * 32, s_);
        tmem_ld32(trow + c_dpt + ch * 32, dp);
        // The piece's 32 chunk rows that this key attends, as bits: rows of
        // the tokens whose window covers the key (a contiguous run), of
        // valid tokens and, when causal, of tokens with sigma(key) <= sigma(q)
        // (the piece's tokens are the same for every lane: broadcast loads).
        uint32_t bits = 0u;
        if (sig_k >= 0) {
          const int r0 = ch * 32;
          const int tq_lo = kpos - P.right - c0, tq_hi = kpos + P.left - c0;
          bits = band_bits(tq_lo * P.g, (tq_hi + 1) * P.g - 1, r0);
          if (bits != 0u) {
            const int t0 = r0 >> P.log2g;
            const int ntok = P.log2g >= 5 ? 1 : (32 >> P.log2g);
            const uint32_t gm = P.log2g >= 5 ? 0xffffffffu : ((1u << P.g) - 1u);
            uint32_t tb = 0u;
            auto tok_ok = [&](int qtk) { return qtk >= 0 && (!kCausal || sig_k <= qtk); };
            if (ntok >= 4) {  // g <= 8: four tokens per load (t0 is a multiple of 4)
              const int4* q4 = reinterpret_cast<const int4*>(qt + t0);
#pragma unroll 1
              for (int i4 = 0; i4 < (ntok >> 2); ++i4) {
                const int4 v4 = q4[i4];
                const int sh = (4 * i4) << P.log2g;
                if (tok_ok(v4.x)) tb |= gm << sh;
                if (tok_ok(v4.y)) tb |= gm << (sh + P.g);
                if (tok_ok(v4.z)) tb |= gm << (sh + 2 * P.g);
                if (tok_ok(v4.w)) tb |= gm << (sh + 3 * P.g);
              }
            } else {
              for (int i = 0; i < ntok; ++i)
                if (tok_ok(qt[t0 + i])) tb |= gm << (i << P.log2g);
            }
            bits &= tb;
          }
        }
        uint32_t pk[16], dk2[16];
        // the rows' lse2' and D four at a time (the same for every lane:
        // broadcast loads)
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const int rb = ch * 32 + 4 * e4;
          const float4 l4 = *reinterpret_cast<const float4*>(cl + rb);
          const float4 d4 = *reinterpret_cast<const float4*>(cd + rb);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
          const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
          float pv[4], dv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const bool ok = (bits >> (4 * e4 + u)) & 1u;
            const float p = ok ? fast_exp2(fmaf(__uint_as_float(s_[4 * e4 + u]), P.scale_log2,
                                                -lv[u]))
                               : 0.f;
            pv[u] = p;
            dv[u] = p * (__uint_as_float(dp[4 * e4 + u]) - dv4[u]);
          }
          pk[2 * e4] = pack_bf16x2(pv[0], pv[1]);
          pk[2 * e4 + 1] = pack_bf16x2(pv[2], pv[3]);
          dk2[2 * e4] = pack_bf16x2(dv[0], dv[1]);
          dk2[2 * e4 + 1] = pack_bf16x2(dv[2], dv[3]);
        }
        tmem_st16(trow + c_st + ch * 32, pk);
        tmem_st16(trow + c_dpt + ch * 32, dk2);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncthreads();
      // dV += P'^T dY, dK += dS^T Q: A from TMEM, B = the chunk's rows (MN-major)
      if (tid == 0) {
        tc_fence_after();
        const uint32_t id = idesc_bf16(kBM, D, 1);
        uint64_t by = sdesc_sw128(sdy, kBM * 128, 1024), bq = sdesc_sw128(sq, kBM * 128, 1024);
        for (int kk = 0; kk < kBM / 16; ++kk) {
          const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
          const uint32_t a = uint32_t((kk >> 1) * 32 + (kk & 1) * 8);  // 16 rows per K step
          umma_bf16_ts(tmem_base + c_dv, tmem_base + c_st + a, by, id, acc);
          umma_bf16_ts(tmem_base + c_dk, tmem_base + c_dpt + a, bq, id, acc);
          by += 128;
          bq += 128;
        }
        umma_commit(bars + 8 * kBarMma);
      }
      if (!cta_wait(bars + 8 * kBarMma, mma_phase, P, abort_flag)) {
        alive = false;
        break;
      }
      mma_phase ^= 1;
      tc_fence_after();
    }
    if (!alive) break;
    {
      // tcgen05.ld is warp-collective: every lane loads, keys of the
      // sequence store.
      const size_t krow_out = (tokb + max(sig_k, 0)) * P.Hkv + kvh;
#pragma unroll 1
      for (int ch = part; ch < D / 32; ch += 2) {
        uint32_t o[32];
        tmem_ld32(trow + c_dv + ch * 32, o);
        if (sig_k >= 0) write_row<D>(P, P.dv, krow_out, o, ch * 32, 1.f);
        tmem_ld32(trow + c_dk + ch * 32, o);
        if (sig_k >= 0) write_row<D>(P, P.dk, krow_out, o, ch * 32, P.scale);
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  cta_teardown(P, bars, tmem_base);
}

// fp32 -> bf16 (the gated merge's accumulated gradients).
__global__ void to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst,
                               size_t n4) {
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n4;
       i += size_t(gridDim.x) * blockDim.x) {
    const float4 f = reinterpret_cast<const float4*>(src)[i];
    reinterpret_cast<uint2*>(dst)[i] = make_uint2(pack_bf16x2(f.x, f.y), pack_bf16x2(f.z, f.w));
  }
}

// ------------------------------------------------------------------ host
struct Layout {  // shared-memory layout of one of the two kernels
  uint32_t off_q, off_dy, off_k, off_v, off_sig, off_col, off_bar, smem;
};
struct Config {
  int Bt, log2g, left, right, span_pad, tmem_alloc;
  Layout dq, dkv;
};

static uint32_t round_up(uint32_t x, uint32_t m) { return (x + m - 1) / m * m; }

static bool make_config(const Problem& pb, Path path, Config& c) {
  if (pb.d != 64 && pb.d != 128) return false;
  if (kBM % pb.g != 0) return false;
  c.Bt = kBM / pb.g;
  c.log2g = 0;
  while ((1 << c.log2g) < pb.g) ++c.log2g;
  if (path == kPathSA) {
    c.left = c.right = pb.window / 2;
  } else {
    c.left = pb.window_swa - 1;
    c.right = 0;
  }
  const long long span = (long long)c.Bt + c.left + c.right;
  if (span > 256) return false;  // S and dP of a query tile side by side in 512 TMEM columns
  c.span_pad = int(round_up(uint32_t(span), 32));
  c.tmem_alloc = 512;
  const uint32_t rowb = uint32_t(pb.d) * 2;
  // qstages: stages of the 128-row Q and dY blocks; kv_rows: K and V rows.
  auto layout = [&](Layout& L, uint32_t qstages, uint32_t kv_rows) {
    L.off_q = 0;
    L.off_dy = L.off_q + qstages * kBM * rowb;
    L.off_k = L.off_dy + qstages * kBM * rowb;
    L.off_v = L.off_k + kv_rows * rowb;
    L.off_sig = L.off_v + kv_rows * rowb;
    L.off_col = round_up(L.off_sig + 4u * (kv_rows + 2 * kBM), 16);
    L.off_bar = round_up(L.off_col + 4u * 6 * kBM, 64);  // dq: 3 x 2 x 128 partials; dkv: 2 x 2 x 128
    L.smem = L.off_bar + 8 * kNumBars + 8 + 1024;
  };
  layout(c.dq, 1, uint32_t(c.span_pad));  // the query tile and its key span
  layout(c.dkv, 2, kBM);                  // two query-chunk stages, the 128-key tile
  return c.dq.smem <= kMaxSmem && c.dkv.smem <= kMaxSmem;
}

static bool device_sm103(int* sms) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (sms) cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  return major == 10 && minor == 3;
}

template <class K>
static cudaError_t launch_k(K kernel, int grid, uint32_t smem, cudaStream_t s, const Params& P) {
  cudaError_t ce = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (ce != cudaSuccess) return ce;
  int resident = 0;
  ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, kernel, kThreads, smem);
  if (ce != cudaSuccess) return ce;
  if (resident < 1) return cudaErrorInvalidConfiguration;
  kernel<<<grid, kThreads, smem, s>>>(P);
  return cudaGetLastError();
}

}  // namespace bwd

bool bwd_supported(const Problem& pb, Path path) {
  if (path != kPathSA && path != kPathSWA) return false;
  if (!bwd::device_sm103(nullptr)) return false;
  bwd::Config c;
  return bwd::make_config(pb, path, c);
}

sa_status_t launch_bwd(const Problem& pb, Path path, const BwdArgs& a, cudaStream_t stream) {
  using namespace bwd;
  int sms = 0;
  if (!device_sm103(&sms)) return fail(SA_ERR_UNSUPPORTED, "device is not sm_103");
  Config c;
  if (!make_config(pb, path, c))
    return fail(SA_ERR_UNSUPPORTED, "window too wide for the backward kernels (key span of a "
                "128-row tile must be <= 256)");
  Params P;
  std::memset(&P, 0, sizeof(P));
  P.q = static_cast<const __nv_bfloat16*>(pb.q);
  P.k = static_cast<const __nv_bfloat16*>(pb.k);
  P.v = static_cast<const __nv_bfloat16*>(pb.v);
  P.dy = static_cast<const __nv_bfloat16*>(a.dout);
  P.perm = (path == kPathSA) ? pb.perm : nullptr;
  P.gate = a.gate;
  P.lse2 = a.lse2;
  P.dsum = a.dsum;
  P.dgate = a.dgate;
  P.dq = a.dq;
  P.dk = a.dk;
  P.dv = a.dv;
  P.out_mode = a.out_mode;
  P.err = pb.err;
  P.B = pb.B;
  P.n = pb.n;
  P.Hq = pb.Hq;
  P.Hkv = pb.Hkv;
  P.g = pb.g;
  P.log2g = c.log2g;
  P.Bt = c.Bt;
  P.left = c.left;
  P.right = c.right;
  P.span_pad = c.span_pad;
  P.causal = (path == kPathSA) ? pb.causal : 0;
  P.scale = pb.scale;
  P.scale_log2 = pb.scale * kLog2e;
  P.tmem_alloc = c.tmem_alloc;
  auto use = [&](const Layout& L) {
    P.off_q = L.off_q;
    P.off_dy = L.off_dy;
    P.off_k = L.off_k;
    P.off_v = L.off_v;
    P.off_sig = L.off_sig;
    P.off_col = L.off_col;
    P.off_bar = L.off_bar;
  };
  P.timeout_cycles = wait_limit_cycles();
  // dQ over query tiles
  use(c.dq);
  P.tiles_per_seq = (pb.n + c.Bt - 1) / c.Bt;
  P.num_tiles = P.tiles_per_seq * pb.B * pb.Hkv;
  int grid = P.num_tiles < sms ? P.num_tiles : sms;
  cudaError_t ce;
  const bool causal = P.causal != 0;
  if (pb.d == 128)
    ce = causal ? launch_k(sa_bwd_dq_kernel<128, true>, grid, c.dq.smem, stream, P)
                : launch_k(sa_bwd_dq_kernel<128, false>, grid, c.dq.smem, stream, P);
  else
    ce = causal ? launch_k(sa_bwd_dq_kernel<64, true>, grid, c.dq.smem, stream, P)
                : launch_k(sa_bwd_dq_kernel<64, false>, grid, c.dq.smem, stream, P);
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "backward dQ launch: %s", cudaGetErrorString(ce));
  // dK, dV over 128-key tiles
  use(c.dkv);
  P.tiles_per_seq = (pb.n + kBM - 1) / kBM;
  P.num_tiles = P.tiles_per_seq * pb.B * pb.Hkv;
  grid = P.num_tiles < sms ? P.num_tiles : sms;
  if (pb.d == 128)
    ce = causal ? launch_k(sa_bwd_dkv_kernel<128, true>, grid, c.dkv.smem, stream, P)
                : launch_k(sa_bwd_dkv_kernel<128, false>, grid, c.dkv.smem, stream, P);
  else
    ce = causal ? launch_k(sa_bwd_dkv_kernel<64, true>, grid, c.dkv.smem, stream, P)
                : launch_k(sa_bwd_dkv_kernel<64, false>, grid, c.dkv.smem, stream, P);
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "backward dK/dV launch: %s", cudaGetErrorString(ce));
  return SA_OK;
}

sa_status_t launch_to_bf16(const float* src, void* dst, size_t count, cudaStream_t stream) {
  const size_t n4 = count / 4;
  const unsigned blocks = unsigned(n4 < 152 * 64 ? (n4 + 255) / 256 : 152 * 16);
  if (n4 > 0)
    bwd::to_bf16_kernel<<<blocks ? blocks : 1, 256, 0, stream>>>(
        src, static_cast<__nv_bfloat16*>(dst), n4);
  const cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "bf16 conversion launch: %s", cudaGetErrorString(ce));
  return SA_OK;
}

}  // namespace sa
