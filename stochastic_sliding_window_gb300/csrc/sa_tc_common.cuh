// Device helpers shared by the tcgen05 kernels: inline PTX wrappers for
// mbarriers, TMA, cp.async, tcgen05 (MMA, TMEM loads, fences), the shared
// memory / instruction descriptors, and the per-row softmax pieces.
#pragma once

#include <cuda.h>  // CUtensorMap (type only)
#include <cuda_bf16.h>
#include <stdint.h>

#include "libsa.h"  // SA_ERRBIT_*

namespace sa {
namespace tcc {

constexpr int kBM = 128;  // MMA M: query rows per tile
// Bound on the final wait for a CTA's own MMAs before TMEM is freed (~2 s at
// the maximum SM clock).  Kept apart from the pipeline wait limit so that a
// short limit never frees TMEM under MMAs still in flight.
constexpr long long kDrainCycles = 4000000000LL;

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// try_wait with a suspend-time hint: the thread sleeps in the instruction
// until the phase completes or about `hint_ns` nanoseconds pass, instead of
// spinning.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity,
                                                   uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  return mbar_try_wait_hint(bar, parity, 1000000u);
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Four arbitrary rows (one 64-element, 128-byte box each) of a 2-D bf16
// tensor into 512 contiguous bytes of smem, 128B-swizzled.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* tm, int col, int r0,
                                            int r1, int r2, int r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(tm), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format:
// start >> 4 in [0,14), LBO >> 4 in [16,30), SBO >> 4 in [32,46),
// version 1 at bit 46, layout SWIZZLE_128B = 2 in [61,64)).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, dense.
// D format [4,6) = 1 (F32); A format [7,10) = 1 (BF16); B format [10,13) = 1;
// B major [16] (1 = MN-major); N >> 3 in [17,23); M >> 4 in [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int nn, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(b_mn_major) << 16) |
         (uint32_t(nn >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane; the wait is in the
// same asm statement so no use of the outputs can be scheduled before it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 16-byte global -> shared copy through L2 only (cp.async.cg).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival counts against the barrier's initial count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Wait on `bar` for the phase of the given parity, for at most `limit`
// SM cycles.  On expiry sets SA_ERRBIT_TIMEOUT in *err and the CTA's abort
// flag; returns false then, or when another role has already aborted.  Each
// sleep in try_wait lasts at most ~limit/4 ns (1 ms at most), so a short
// limit is honoured even while the phase never completes.
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, long long limit,
                                             int32_t* err, volatile int* abort_flag) {
  const uint32_t hint = limit >= 4000000LL ? 1000000u : uint32_t(limit > 4 ? limit >> 2 : 1);
  if (mbar_try_wait_hint(bar, parity, hint)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_hint(bar, parity, hint)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      atomicOr(err, SA_ERRBIT_TIMEOUT);
      return false;
    }
  }
}

// 2^x on the SFU (ex2.approx.ftz.f32); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Issue a 32-column TMEM load without waiting; pair with tmem_wait_ld()
// followed by reg_fence() on every destination before the values are used.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Maximum of 32 consecutive fp32 columns of this thread's TMEM lane, taken by
// the loads themselves (tcgen05.ld.red, an sm_103 form: the load returns the
// max of the elements it read beside the elements).  The elements are not
// used.  Two 16-column loads, one wait (a 32-column ld.red made ptxas spill).
#pragma nv_diag_suppress 550  // a and b are written and deliberately unused
__device__ __forceinline__ float tmem_max32(uint32_t taddr) {
  uint32_t a[16], b[16];
  float m0, m1;
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15}, %16, [%17];"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
        "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]),
        "=r"(a[14]), "=r"(a[15]), "=f"(m0)
      : "r"(taddr)
      : "memory");
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15}, %16, [%17];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]),
        "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]),
        "=r"(b[14]), "=r"(b[15]), "=f"(m1)
      : "r"(taddr + 16)
      : "memory");
  return fmaxf(m0, m1);
}
#pragma nv_diag_default 550
// Orders every later use of r after the preceding tmem_wait_ld().
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i]));
}

// Packed pairs of fp32 (sm_100 family f32x2 arithmetic): each lane of the
// pair is rounded exactly as the scalar instruction would round it.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t x) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(x));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Columns c0 .. c0+31 that fall in the band [lo, hi], as bits (bit e:
// column c0 + e).
__device__ __forceinline__ uint32_t band_bits(int lo, int hi, int c0) {
  const int a = lo - c0, b = hi - c0;  // first and last allowed offsets
  if (b < 0 || a > 31 || a > b) return 0u;
  const uint32_t upto_b = b >= 31 ? 0xffffffffu : ((2u << b) - 1u);
  const uint32_t from_a = a <= 0 ? 0xffffffffu : ~((1u << a) - 1u);
  return upto_b & from_a;
}

// Row sums of p are accumulated in one fixed order by every tcgen05 kernel
// (so that kernels subtracting the same reference agree bit for bit): pair
// e2 of a 32-column chunk adds p[2 e2] to acc[2 (e2 & 1)] and p[2 e2 + 1] to
// acc[2 (e2 & 1) + 1]; the row sum is (acc[0] + acc[1]) + (acc[2] + acc[3]).

// Per-row state of one tile, shared by the softmax variants.
struct RowCtx {
  int lo, hi;      // attended column band of this row (sequence ends folded in)
  int wlo, whi;    // band that holds for every row of the warp
  int sig_p;       // original index of this row's query token
  float scale_log2;
};

// Mask one 32-column chunk in registers: out-of-band and (causal) later
// tokens become -inf.  Returns the chunk's masked maximum.
template <bool kCausal>
__device__ __forceinline__ float mask_chunk(uint32_t (&v)[32], const int32_t* sig, int c0,
                                            const RowCtx& rc) {
  const bool need_band = !(c0 >= rc.wlo && c0 + 31 <= rc.whi);  // warp-uniform
  float m0 = -INFINITY, m1 = -INFINITY;
  const int4* sg4 = reinterpret_cast<const int4*>(sig + c0);
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    int sv[4] = {0, 0, 0, 0};
    if (kCausal) {
      const int4 q4 = sg4[e4];
      sv[0] = q4.x; sv[1] = q4.y; sv[2] = q4.z; sv[3] = q4.w;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + e4 * 4 + u;
      bool ok = kCausal ? (sv[u] <= rc.sig_p) : true;
      if (need_band) ok = ok && (c >= rc.lo) && (c <= rc.hi);
      const float x = ok ? __uint_as_float(v[e4 * 4 + u]) : -INFINITY;
      v[e4 * 4 + u] = __float_as_uint(x);
      if (u & 1) m1 = fmaxf(m1, x); else m0 = fmaxf(m0, x);
    }
  }
  return fmaxf(m0, m1);
}

// Mask one 32-column chunk given the row's causal bits for it (bit e set:
// column c0+e is allowed) and the band: excluded columns become -inf.
// Returns the chunk's masked maximum.
__device__ __forceinline__ float mask_chunk_bits(uint32_t (&v)[32], uint32_t bits, int c0,
                                                 const RowCtx& rc) {
  const bool need_band = !(c0 >= rc.wlo && c0 + 31 <= rc.whi);  // warp-uniform
  if (need_band) {
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int c = c0 + e;
      if (c < rc.lo || c > rc.hi) bits &= ~(1u << e);
    }
  }
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float x = (bits >> e) & 1u ? __uint_as_float(v[e]) : -INFINITY;
    v[e] = __float_as_uint(x);
    if (e & 1) m1 = fmaxf(m1, x); else m0 = fmaxf(m0, x);
  }
  return fmaxf(m0, m1);
}

// p = 2^(s * scale * log2 e - max) for one masked chunk; bf16 P to smem in
// the K-major 128B-swizzled layout the PV MMA reads; adds to the row sums.
__device__ __forceinline__ void exp_store_chunk(const uint32_t (&v)[32], float ms, float sl2,
                                                uint8_t* pbase, int r, int c0, float (&acc)[4]) {
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    uint32_t pk[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      const float p0 = fast_exp2(fmaf(__uint_as_float(v[q4 * 8 + 2 * e2]), sl2, -ms));
      const float p1 = fast_exp2(fmaf(__uint_as_float(v[q4 * 8 + 2 * e2 + 1]), sl2, -ms));
      acc[2 * (e2 & 1)] += p0;
      acc[2 * (e2 & 1) + 1] += p1;
      pk[e2] = pack_bf16x2(p0, p1);
    }
    const int col8 = c0 + q4 * 8;
    const int kb = col8 >> 6;
    const int c16 = (col8 & 63) >> 3;
    uint4* dst = reinterpret_cast<uint4*>(pbase + kb * (kBM * 128) + r * 128 +
                                          ((c16 ^ (r & 7)) << 4));
    *dst = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

// One SA output row computed exactly by one thread on its own, from global
// memory: the row of position p (query token sig_p) at output row `orow`.
// fp32 scores against the keys of the band [p - left, p + right] within
// [0, n) that the row attends (sigma(q) <= sigma(p) when causal), their
// maximum, the softmax and the weighted sum of V rows, then the gate and the
// accumulation as the tensor-core epilogues apply them.  The tensor-core
// kernels take their softmax reference from every key column they hold,
// attended or not; this is the path of a row whose attended maximum lies so
// far below that reference that its p underflow (a row sum below 2^-60),
// which ordinary inputs never produce.  Kept out of line.
struct ExactRow {
  const __nv_bfloat16* q;   // [B, n, Hq, d]
  const __nv_bfloat16* k;   // [B, n, Hkv, d]
  const __nv_bfloat16* v;
  const int32_t* perm_b;    // sigma of this batch row, or nullptr (identity)
  const float* gate;        // logits [B, n, Hq] or nullptr
  __nv_bfloat16* out;
  size_t orow, kv0;         // output (= query) row; b * n
  int n, Hkv, kvh, p, sig_p, left, right, causal, accumulate;
  float scale_log2;
};

template <int D>
__device__ __noinline__ void exact_row(const ExactRow r) {
  const __nv_bfloat16* qr = r.q + r.orow * D;
  const int q_lo = max(r.p - r.left, 0), q_hi = min(r.p + r.right, r.n - 1);
  auto key_token = [&](int pos) { return r.perm_b ? r.perm_b[pos] : pos; };
  auto attended = [&](int tok) {
    return unsigned(tok) < unsigned(r.n) && !(r.causal && tok > r.sig_p);
  };
  auto score = [&](int tok) {
    const __nv_bfloat16* kr = r.k + ((r.kv0 + tok) * r.Hkv + r.kvh) * D;
    float s = 0.f;
    for (int e = 0; e < D; ++e) s = fmaf(__bfloat162float(qr[e]), __bfloat162float(kr[e]), s);
    return s * r.scale_log2;
  };
  float m = -INFINITY;
  for (int pos = q_lo; pos <= q_hi; ++pos) {
    const int tok = key_token(pos);
    if (attended(tok)) m = fmaxf(m, score(tok));
  }
  float mul = 1.f;
  if (r.gate != nullptr) mul = 1.f / (1.f + expf(-r.gate[r.orow]));
  __nv_bfloat16* op = r.out + r.orow * D;
  // 32 output columns at a time (registers, no local array); the weights
  // are recomputed for each block
  for (int e0 = 0; e0 < D; e0 += 32) {
    float y[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) y[e] = 0.f;
    float l = 0.f;
    for (int pos = q_lo; pos <= q_hi; ++pos) {
      const int tok = key_token(pos);
      if (!attended(tok)) continue;
      const float w = exp2f(score(tok) - m);
      l += w;
      const __nv_bfloat16* vr = r.v + ((r.kv0 + tok) * r.Hkv + r.kvh) * D + e0;
#pragma unroll
      for (int e = 0; e < 32; ++e) y[e] = fmaf(w, __bfloat162float(vr[e]), y[e]);
    }
    const float f = l > 0.f ? mul / l : 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      float o = y[e] * f;
      if (r.accumulate) o += __bfloat162float(op[e0 + e]);
      op[e0 + e] = __float2bfloat16(o);
    }
  }
}

}  // namespace tcc
}  // namespace sa
