// tcgen05 kernel for SA / SWA with wide windows: each tile's key span is
// streamed through shared memory in chunks of 128 keys, with an online
// softmax.
//
// Same attention as the other tcgen05 kernels (Stochastic Attention summary,
// "Core mechanism" steps 1-3; causal rule from "Theoretical properties"; SWA
// from "Problem statement"): a tile here is 2*Bt = 256/g consecutive permuted
// positions of one (sequence, kv head) pair stacked with the g query heads of
// that kv head (256 rows, r = t*g + j: two M = 128 halves), over its key span
// [p0 - left, p0 + 2*Bt - 1 + right].  The span is cut into chunks of 128
// keys, each loaded once for both halves.  Per chunk and half, S = Q K^T lands
// in the half's TMEM buffer; the half's softmax warpgroup masks it (window
// band and, when causal, sigma[q] <= sigma[p]), keeps a running reference
// maximum (from the chunks' maxima over every key column, returned by the
// TMEM loads) and sum per row and writes bf16 P over S; O += P V accumulates
// in the half's TMEM accumulator.  A row's reference maximum is raised -- and
// O and the sum rescaled by 2^(old - new) -- only when a chunk's maximum
// exceeds it by more than 2^8, so most chunks need no correction of O.  Shared
// memory does not grow with the window: any window fits.
//
// Roles (four warpgroups, 512 threads):
//   warps 0-6  producers: cp.async of the 256 Q rows of a tile and of the 128
//               K and V rows of each chunk (with the chunk's key tokens)
//   warp 7      lane 0 issues S = Q K^T of each half and chunk as soon as its
//               operands are ready; the warp owns TMEM
//   warps 8-11  softmax, O correction, O += P V issue and epilogue of rows
//               0-127 (one thread of the warpgroup issues the O MMAs, so no
//               other warp has to notice that P is ready)
//   warps 12-15 the same for rows 128-255
// Every wait is bounded (SA_ERRBIT_TIMEOUT); producer copies are drained
// before exit.
#include "sa_internal.h"
#include "sa_tc_common.cuh"

#include <cstring>

namespace sa {
namespace chunk {

using namespace tcc;

constexpr int kThreads = 512;
constexpr int kProducers = 224;  // warps 0-6
constexpr int kMmaWarp = 7;
constexpr int kFirstSoftmaxWarp = 8;
constexpr int kLaunchRegs = 128;
constexpr int kCtrlRegs = 96;
constexpr int kSoftmaxRegs = 160;
static_assert(256 * kCtrlRegs + 256 * kSoftmaxRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kRows = 2 * kBM;      // rows of a tile: two halves of M = 128
constexpr int kKC = 128;            // keys per chunk
constexpr int kSub = kKC / 32;      // 32-column pieces of a chunk
constexpr int kMaxRows = 10;        // rows per producer thread per chunk
constexpr int kBatch = 8;           // Q rows whose tokens are loaded before their copies
constexpr float kRescaleLog2 = 8.f; // raise a row's reference maximum past 2^8
constexpr uint32_t kMaxSmem = 232448;

struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* perm;  // [B, n]; nullptr: identity (SWA)
  const float* gate;    // [B, n, Hq] logits or nullptr
  __nv_bfloat16* out;
  int32_t* err;
  int B, n, Hq, Hkv, g, log2g, Bt;
  int left, right, nchunks;
  int qstages;  // Q tile stages: 2 when shared memory allows (d = 64), else 1
  int causal, accumulate;
  float scale_log2;
  int tiles_per_seq, num_tiles;
  uint32_t q_bytes, kv_bytes;  // one half (128 rows) of the Q tile; one K (or V) chunk
  uint32_t off_k, off_v, off_csig, off_qtok, off_bits, off_bar;
  int tmem_alloc;
  long long timeout_cycles;
};

// Barrier slots (8 bytes each) after off_bar.  Chunk stages are indexed by
// the CTA-local chunk number c_all & 1 (c_all = x * nchunks + chunk); [2]
// half families by the half (softmax warpgroup) h.
enum : uint32_t {
  kQfull = 0,    // [stage] Q rows and tokens of tile x landed (cp.async)
  kQfree = 2,    // [stage] both halves' last S MMA of tile x done and every softmax warp
                 // has read the tile's tokens: the stage is free
  kCfull = 4,    // [2] K, V rows and key tokens of chunk c_all landed
  kCfree = 6,    // [2] both halves' O MMA of chunk c_all done: its stage is free
  kSfull = 8,    // [h] S of the half's current chunk in its TMEM buffer
  kPfull = 10,   // [h] P of the half's current chunk written (4 softmax warps)
  kPVdone = 12,  // [h] the half's O MMA of its current chunk done
  kOfull = 14,   // [h] the half's last O MMA of tile x done
  kOfree = 16,   // [h] the half's epilogue has read O of tile x (4 warps)
  kDrain = 18,
  kDrainH = 19,  // [h] final completion of the half's O MMAs
  kNumBars = 21,
};

struct Tile {
  int b, kvh, p0;
};
__device__ __forceinline__ Tile tile_of(const Params& P, int tile) {
  const int s = tile / P.tiles_per_seq;
  Tile t;
  t.p0 = (tile - s * P.tiles_per_seq) * P.Bt;
  t.b = s / P.Hkv;
  t.kvh = s - t.b * P.Hkv;
  return t;
}

__device__ __forceinline__ void cta_range(const Params& P, int& begin, int& end) {
  begin = int((long long)blockIdx.x * P.num_tiles / gridDim.x);
  end = int((long long)(blockIdx.x + 1) * P.num_tiles / gridDim.x);
}

// 4-byte global -> shared copy (the tokens the softmax warps read).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

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

// A from TMEM (P), B from shared memory (V), D in TMEM (O).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32-byte global store: one whole sector per thread.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&r)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// ------------------------------------------------------------------ producers
template <int D>
__device__ void producer_role(const Params& P, uint8_t* smem, uint32_t sbase, uint32_t bars,
                              volatile int* abort_flag, volatile int* vote) {
  constexpr int CPR = D / 8;             // 16-byte chunks per row
  constexpr int RPP = kProducers / CPR;  // rows per pass of the producers
  static_assert((kKC + RPP - 1) / RPP <= kMaxRows, "rows per thread");
  const int tid = threadIdx.x;
  const int cc = tid % CPR;
  const int r_first = tid / CPR;
  const int kb = cc >> 3, c8 = cc & 7;
  auto wait = [&](uint32_t bar, uint32_t par) {
    return bounded_wait(bar, par, P.timeout_cycles, P.err, abort_flag);
  };
  auto agree = [&](bool ok) {
    if (tid == 0) *vote = ok ? 1 : 0;
    asm volatile("bar.sync 1, %0;" ::"n"(kProducers) : "memory");
    const bool v = *vote != 0;
    asm volatile("bar.sync 1, %0;" ::"n"(kProducers) : "memory");  // vote read by all
    return v;
  };
  auto token = [&](const Tile& t, int pos) {  // sigma of position pos (clamped)
    const int qc = min(max(pos, 0), P.n - 1);
    int tok = P.perm ? __ldg(P.perm + size_t(t.b) * P.n + qc) : qc;
    if (unsigned(tok) >= unsigned(P.n)) {
      atomicOr(P.err, SA_ERRBIT_RANGE);
      tok = 0;
    }
    return tok;
  };
  int begin, end;
  cta_range(P, begin, end);
  const int ntiles = end - begin;
  const int nch = P.nchunks;
  const size_t tokstride = size_t(P.Hq) * D;
  int tk[kMaxRows];  // tokens of this thread's rows of the next chunk
  auto fetch_chunk = [&](int call) {
    const int x = call / nch, c = call - (call / nch) * nch;
    const Tile t = tile_of(P, begin + x);
    const int k0 = t.p0 - P.left + c * kKC;
#pragma unroll
    for (int k = 0; k < kMaxRows; ++k) {
      const int i = r_first + RPP * k;
      if (i < kKC) tk[k] = token(t, k0 + i);
    }
  };
  if (ntiles > 0) fetch_chunk(0);
  for (int x = 0; x < ntiles; ++x) {
    const Tile t = tile_of(P, begin + x);
    const int qs = x % P.qstages;
    // The Q stage is free once both halves' last S MMA of its previous tile
    // (x - qstages) is done.
    bool ok = true;
    if (tid == 0 && x >= P.qstages)
      ok = wait(bars + 8 * (kQfree + qs), uint32_t(x / P.qstages - 1) & 1u);
    if (!agree(ok)) break;
    const uint32_t qstage = sbase + uint32_t(qs) * 2 * P.q_bytes;
    {
      // 256 rows (r = t*g + j) in two halves of [128 rows x D], each two
      // K-blocks of [128 rows x 128 B], swizzled.
      const __nv_bfloat16* qbase =
          P.q + (size_t(t.b) * P.n * P.Hq + size_t(t.kvh) * P.g) * D + cc * 8;
      for (int r0 = r_first; r0 < kRows; r0 += RPP * kBatch) {
        int tq[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int r = r0 + RPP * k;
          if (r < kRows) tq[k] = token(t, t.p0 + (r >> P.log2g));
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int r = r0 + RPP * k;
          if (r < kRows)
            cp_async16(qstage + uint32_t(r >> 7) * P.q_bytes + kb * (kBM * 128) + (r & 127) * 128 +
                           ((c8 ^ (r & 7)) << 4),
                       qbase + tq[k] * tokstride + (r & (P.g - 1)) * D);
        }
      }
      if (P.perm) {  // the tile's tokens, for the softmax warps
        for (int i = tid; i < P.Bt; i += kProducers) {
          const int qc = min(t.p0 + i, P.n - 1);
          cp_async4(sbase + P.off_qtok + uint32_t(qs * kRows + i) * 4, P.perm + size_t(t.b) * P.n + qc);
        }
      }
      cp_async_arrive_noinc(bars + 8 * (kQfull + qs));
    }
    for (int c = 0; c < nch; ++c) {
      const int call = x * nch + c;
      const int s = call & 1;
      // The stage's previous chunk (call - 2) must have had both halves' O MMAs.
      ok = true;
      if (tid == 0 && call >= 2) ok = wait(bars + 8 * (kCfree + s), uint32_t((call >> 1) - 1) & 1u);
      if (!agree(ok)) {
        x = ntiles;
        break;
      }
      const int k0 = t.p0 - P.left + c * kKC;
      const uint32_t sk = sbase + P.off_k + uint32_t(s) * P.kv_bytes + kb * (kKC * 128);
      const uint32_t sv = sbase + P.off_v + uint32_t(s) * P.kv_bytes + kb * (kKC * 128);
      const size_t rowbase = size_t(t.b) * P.n;
#pragma unroll
      for (int k = 0; k < kMaxRows; ++k) {
        const int i = r_first + RPP * k;
        if (i < kKC) {
          const size_t off = ((rowbase + tk[k]) * P.Hkv + t.kvh) * D + cc * 8;
          const uint32_t d = i * 128 + ((c8 ^ (i & 7)) << 4);
          cp_async16(sk + d, P.k + off);
          cp_async16(sv + d, P.v + off);
          if (P.perm && cc == 0) {  // the chunk's key tokens, for the masks
            const int qc = min(max(k0 + i, 0), P.n - 1);
            cp_async4(sbase + P.off_csig + uint32_t(s * kKC + i) * 4, P.perm + rowbase + qc);
          }
        }
      }
      cp_async_arrive_noinc(bars + 8 * (kCfull + s));
      if (call + 1 < ntiles * nch) fetch_chunk(call + 1);  // loaded now, used next
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // own copies land before exit
}

// ------------------------------------------------------------------ MMA issue
template <int D>
__device__ void mma_role(const Params& P, uint32_t sbase, uint32_t tmem_base, uint32_t bars,
                         volatile int* abort_flag) {
  int begin, end;
  cta_range(P, begin, end);
  const int nch = P.nchunks;
  const int total = (end - begin) * nch;
  const uint32_t idesc_qk = idesc_bf16(kBM, kKC, 0);
  // S of half h in TMEM columns [h*128, h*128 + 128); O of half h at 256 + h*D.
  // Shared-memory descriptors of every stage, built once (kept in registers:
  // chosen by selects, not indexed).
  const uint64_t q00 = sdesc_sw128(sbase, 16, 1024);
  const uint64_t q01 = sdesc_sw128(sbase + P.q_bytes, 16, 1024);
  const uint64_t q10 = sdesc_sw128(sbase + 2 * P.q_bytes, 16, 1024);
  const uint64_t q11 = sdesc_sw128(sbase + 3 * P.q_bytes, 16, 1024);
  const uint64_t k0 = sdesc_sw128(sbase + P.off_k, 16, 1024);
  const uint64_t k1 = sdesc_sw128(sbase + P.off_k + P.kv_bytes, 16, 1024);
  // c: the chunk within its tile; qs: the tile's Q stage.
  auto qk = [&](int h, int call, int c, int qs) {
    fence_proxy_async_smem();  // cp.async (generic proxy) data -> tensor core reads
    tc_fence_after();
    const uint32_t d = tmem_base + uint32_t(h * kKC);
    const uint64_t a0 = qs == 0 ? (h == 0 ? q00 : q01) : (h == 0 ? q10 : q11);
    const uint64_t b0 = (call & 1) ? k1 : k0;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint64_t da = uint64_t((kk >> 2) * (kBM * 128 / 16) + (kk & 3) * 2);
      const uint64_t db = uint64_t((kk >> 2) * (kKC * 128 / 16) + (kk & 3) * 2);
      umma_bf16(d, a0 + da, b0 + db, idesc_qk, kk > 0 ? 1u : 0u);
    }
    umma_commit(bars + 8 * (kSfull + h));
    if (c == nch - 1) umma_commit(bars + 8 * (kQfree + qs));
  };
  // Per half: QK of chunk call once its K rows have landed and the half's
  // previous O MMA (issued by the half's softmax warpgroup) has read P out of
  // the S buffer.  Chunk and Q stage of each half's next QK are kept as
  // counters: this single thread's loop stays free of divisions, which would
  // delay every reaction to a barrier.
  int qn[2] = {0, 0};
  int qc[2] = {0, 0};                    // QK: chunk
  int qst[2] = {0, 0}, qph[2] = {0, 0};  // QK: Q stage and its parity
  long long last = clock64();
  while (qn[0] < total || qn[1] < total) {
    bool progress = false;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (qn[h] < total) {
        const int call = qn[h];
        bool ready = mbar_test_wait(bars + 8 * (kCfull + (call & 1)), (call >> 1) & 1) &&
                     mbar_test_wait(bars + 8 * (kPVdone + h), (call & 1) ^ 1);
        if (ready && qc[h] == 0) ready = mbar_test_wait(bars + 8 * (kQfull + qst[h]), qph[h]);
        if (ready) {
          qk(h, call, qc[h], qst[h]);
          ++qn[h];
          if (++qc[h] == nch) {
            qc[h] = 0;
            if (++qst[h] == P.qstages) {
              qst[h] = 0;
              qph[h] ^= 1;
            }
          }
          progress = true;
        }
      }
    }
    if (progress) {
      last = clock64();
    } else {
      if (*abort_flag) break;
      if (clock64() - last > P.timeout_cycles) {
        *abort_flag = 1;
        atomicOr(P.err, SA_ERRBIT_TIMEOUT);
        break;
      }
      __nanosleep(20);
    }
  }
  umma_commit(bars + 8 * kDrain);
  const long long t0 = clock64();
  while (!mbar_try_wait(bars + 8 * kDrain, 0) && clock64() - t0 < kDrainCycles) {
  }
}

// ------------------------------------------------------------------ softmax
template <int D, bool kCausal>
__device__ void softmax_role(const Params& P, uint8_t* smem, uint32_t sbase, uint32_t tmem_base,
                             uint32_t bars, volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = (warp - kFirstSoftmaxWarp) >> 2;  // the half of the tile (rows h*128 ..)
  const int quad = warp & 3;
  const int wi = h * 4 + quad;  // this warp among the eight softmax warps
  const int r = h * kBM + quad * 32 + lane;
  const int t = r >> P.log2g;
  const int j = r & (P.g - 1);
  const int tpw = 32 >> P.log2g;                   // tokens of this warp's rows:
  const int tw0 = (h * kBM + quad * 32) >> P.log2g;  // tw0 .. tw0 + tpw - 1
  const uint32_t lanes = uint32_t(quad * 32) << 16;
  const uint32_t o_taddr = tmem_base + lanes + uint32_t(2 * kKC + h * D);
  const int32_t* qtok = reinterpret_cast<const int32_t*>(smem + P.off_qtok);
  const int32_t* csig = reinterpret_cast<const int32_t*>(smem + P.off_csig);
  uint32_t* wall = reinterpret_cast<uint32_t*>(smem + P.off_bits) + wi * (2 * 32 * kSub);
  // this warp's tokens (sigma of its rows' positions) for the causal masks
  int32_t* wsig = reinterpret_cast<int32_t*>(smem + P.off_bits + 8 * 2 * 32 * kSub * 4) + wi * 32;
  auto wwait = [&](uint32_t bar, uint32_t par) {
    const bool ok = bounded_wait(bar, par, P.timeout_cycles, P.err, abort_flag);
    return __all_sync(0xffffffffu, ok);
  };
  int begin, end;
  cta_range(P, begin, end);
  const int ntiles = end - begin;
  const int nch = P.nchunks;
  const uint64_t sl2 = f2_pack(P.scale_log2, P.scale_log2);
  const bool issuer = quad == 0 && lane == 0;  // issues this half's O MMAs
  const uint32_t idesc_pv = idesc_bf16(kBM, D, 1);
  bool issued = false;
  bool alive = true;
  for (int x = 0; x < ntiles && alive; ++x) {
    const Tile tl = tile_of(P, begin + x);
    const int qs = x % P.qstages;
    if (!wwait(bars + 8 * (kQfull + qs), uint32_t(x / P.qstages) & 1u)) break;
    // Tokens of this warp's rows, kept in registers: the Q stage (and its
    // token list) is refilled as soon as the tile's last S MMAs are done.
    int wtok = 0;
    if (lane < tpw) {
      const int tt = tw0 + lane;
      wtok = P.perm ? qtok[qs * kRows + tt] : min(tl.p0 + tt, P.n - 1);
    }
    const int sig_p = __shfl_sync(0xffffffffu, wtok, t - tw0);
    __syncwarp();  // the previous tile's reads of wsig are done
    if (lane < tpw) wsig[lane] = wtok;
    __syncwarp();
    // The Q stage's tokens are read: with one chunk per tile the tile's only
    // S MMAs can be done before this warp gets here, so the stage is refilled
    // only once every softmax warp has also arrived.
    if (lane == 0) mbar_arrive(bars + 8 * (kQfree + qs));
    bool row_valid = tl.p0 + t < P.n;
    if (row_valid && unsigned(sig_p) >= unsigned(P.n)) {
      atomicOr(P.err, SA_ERRBIT_RANGE);
      row_valid = false;
    }
    float ms_ref = -INFINITY;  // reference maximum of the row's p (scaled, log2)
    float l = 0.f;
    for (int c = 0; c < nch; ++c) {
      const int call = x * nch + c;
      const int b = call & 1;  // chunk stage
      if (!wwait(bars + 8 * (kCfull + b), uint32_t(call >> 1) & 1u)) {  // the chunk's key tokens
        alive = false;
        break;
      }
      // Mask words of the chunk for this warp's tokens: bit e of word
      // (token, q) set iff key column c*128 + 32q + e is attended.
      uint32_t* wb = wall + b * (32 * kSub);
      // (consecutive lanes take consecutive tokens of one piece, so the
      // piece's key tokens are broadcast loads)
      for (int w = lane; w < tpw * kSub; w += 32) {
        const int q = w / tpw, ti = w - q * tpw;
        const int tt = tw0 + ti;
        const int lo = max(tt, P.left - tl.p0) - c * kKC - 32 * q;
        const int hi = (tl.p0 + tt < P.n ? min(tt + P.left + P.right, P.n - 1 - tl.p0 + P.left)
                                         : -1 - kKC * nch) -
                       c * kKC - 32 * q;
        uint32_t word = band_bits(lo, hi, 0);
        if (kCausal && word != 0u) {
          const int sp = wsig[ti];
          const int4* s4p = reinterpret_cast<const int4*>(csig + b * kKC + 32 * q);
          uint32_t cw = 0;
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const int4 s4 = s4p[e4];
            cw |= (s4.x <= sp ? 1u : 0u) << (4 * e4);
            cw |= (s4.y <= sp ? 1u : 0u) << (4 * e4 + 1);
            cw |= (s4.z <= sp ? 1u : 0u) << (4 * e4 + 2);
            cw |= (s4.w <= sp ? 1u : 0u) << (4 * e4 + 3);
          }
          word &= cw;
        }
        wb[ti * kSub + q] = word;
      }
      __syncwarp();
      const uint32_t* wrow = wb + (t - tw0) * kSub;
      if (!wwait(bars + 8 * (kSfull + h), uint32_t(call) & 1u)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const uint32_t sb = tmem_base + lanes + uint32_t(h * kKC);
      // pass 1: the chunk's maximum over all its 128 key columns, attended
      // or not, returned by the TMEM loads themselves (no mask test).  Every
      // column holds a real key of this launch (positions past either end
      // load a clamped token's rows), so the reference below is finite and
      // never below the row's attended maximum; a reference so far above it
      // that the attended p underflow shows as a row sum below 2^-60, and
      // that row is recomputed exactly (exact_row).
      float mx = -INFINITY;
#pragma unroll 1
      for (int q = 0; q < kSub; ++q) mx = fmaxf(mx, tmem_max32(sb + q * 32));
      // online reference: rescale only when the maximum grows past 2^8
      float alpha = 1.f;
      bool rescale = false;
      if (mx != -INFINITY) {
        const float msc = mx * P.scale_log2;
        if (ms_ref == -INFINITY) {
          ms_ref = msc;  // the row's first chunk: O and l are still 0
        } else if (msc > ms_ref + kRescaleLog2) {
          alpha = fast_exp2(ms_ref - msc);
          ms_ref = msc;
          l *= alpha;
          rescale = true;
        }
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O must hold the O MMAs of every earlier chunk of the tile.
        if (c > 0 && !wwait(bars + 8 * (kPVdone + h), uint32_t(call - 1) & 1u)) {
          alive = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(o_taddr + q * 32, o);
          uint32_t lo16[16], hi16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            lo16[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            hi16[e] = __float_as_uint(__uint_as_float(o[16 + e]) * alpha);
          }
          tmem_st16(o_taddr + q * 32, lo16);
          tmem_st16(o_taddr + q * 32 + 16, hi16);
        }
        tmem_wait_st();
      }
      // pass 2: p = 2^(s*scale*log2e - ref) on attended keys, bf16 P over S
      const float nref = ms_ref == -INFINITY ? 0.f : -ms_ref;
      const uint64_t nms = f2_pack(nref, nref);
      uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll 1
      for (int q = 0; q < kSub; ++q) {
        uint32_t v[32];
        tmem_ld32(sb + q * 32, v);
        const uint32_t bits = wrow[q];
        uint32_t pk[16];
#pragma unroll
        for (int e2 = 0; e2 < 16; ++e2) {
          const float2 y = f2_unpack(f2_fma(f2_pack(__uint_as_float(v[2 * e2]),
                                                    __uint_as_float(v[2 * e2 + 1])),
                                            sl2, nms));
          const float p0 = (bits >> (2 * e2)) & 1u ? fast_exp2(y.x) : 0.f;
          const float p1 = (bits >> (2 * e2 + 1)) & 1u ? fast_exp2(y.y) : 0.f;
          acc2[e2 & 1] = f2_add(acc2[e2 & 1], f2_pack(p0, p1));
          pk[e2] = pack_bf16x2(p0, p1);
        }
        tmem_st16(sb + q * 16, pk);
      }
      const float2 a01 = f2_unpack(acc2[0]), a23 = f2_unpack(acc2[1]);
      l += (a01.x + a01.y) + (a23.x + a23.y);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8 * (kPfull + h));
      // Once all four warps have written P, one thread issues O += P V (A = P
      // from the half's S buffer, B = V of the chunk's stage).  The chunk's V
      // rows landed with its keys (kCfull, waited above).  The tile's first O
      // MMA overwrites O: every warp of the half read O of the previous tile
      // before it wrote this P, which the P barrier orders.
      if (issuer && bounded_wait(bars + 8 * (kPfull + h), uint32_t(call) & 1u, P.timeout_cycles,
                                 P.err, abort_flag)) {
        tc_fence_after();
        const uint32_t sbuf = tmem_base + uint32_t(h * kKC);
        const uint32_t o = tmem_base + uint32_t(2 * kKC + h * D);
        uint64_t bd = sdesc_sw128(sbase + P.off_v + uint32_t(b) * P.kv_bytes, kKC * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < kKC / 16; ++kk) {
          umma_bf16_ts(o, sbuf + 8 * kk, bd, idesc_pv, (c > 0 || kk > 0) ? 1u : 0u);
          bd += 128;  // 16 keys of 128 B
        }
        umma_commit(bars + 8 * (kPVdone + h));
        umma_commit(bars + 8 * (kCfree + b));
        if (c == nch - 1) umma_commit(bars + 8 * (kOfull + h));
        issued = true;
      }
    }
    if (!alive) break;

    // epilogue: O / l (x sigmoid(gate)), scattered to row sigma[p0 + t]
    if (!wwait(bars + 8 * (kOfull + h), uint32_t(x & 1))) break;
    tc_fence_after();
    // l is at least the row's largest attended p, 2^-(reference - attended
    // maximum) (every valid row attends its own key): l < 2^-60 means that
    // gap is above 60, and the row is computed exactly instead
    const bool exact = row_valid && l < 0x1p-60f;
    float mul = l > 0.f ? 1.f / l : 0.f;
    const size_t orow =
        row_valid ? (size_t(tl.b) * P.n + sig_p) * P.Hq + size_t(tl.kvh) * P.g + j : 0;
    if (P.gate != nullptr && row_valid) mul *= 1.f / (1.f + expf(-P.gate[orow]));
    // O leaves TMEM in 64-column halves (fewer registers held at once); the
    // accumulator is handed back once the last half is read.
    const uint64_t mul2 = f2_pack(mul, mul);
    __nv_bfloat16* op = P.out + orow * D;
#pragma unroll 1
    for (int hf = 0; hf < D / 64; ++hf) {
      uint32_t o[2][32];
      tmem_ld32_async(o_taddr + hf * 64, o[0]);
      tmem_ld32_async(o_taddr + hf * 64 + 32, o[1]);
      tmem_wait_ld();
      reg_fence(o[0]);
      reg_fence(o[1]);
      if (hf == D / 64 - 1) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (kOfree + h));
      }
      if (row_valid && !exact) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t pk[8];
            float f[16];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int k = half * 16 + 2 * e;
              const float2 y = f2_unpack(f2_mul(f2_pack(__uint_as_float(o[q][k]),
                                                        __uint_as_float(o[q][k + 1])),
                                                mul2));
              f[2 * e] = y.x;
              f[2 * e + 1] = y.y;
            }
            __nv_bfloat16* dst = op + hf * 64 + q * 32 + half * 16;
            if (P.accumulate) {  // second pass of the gated sum: add the row there
              const uint4* src = reinterpret_cast<const uint4*>(dst);
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                const uint4 pv4 = src[h2];
                const __nv_bfloat162* pv2 = reinterpret_cast<const __nv_bfloat162*>(&pv4);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 pf = __bfloat1622float2(pv2[e]);
                  f[8 * h2 + 2 * e] += pf.x;
                  f[8 * h2 + 2 * e + 1] += pf.y;
                }
              }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
            st_global_v8(dst, pk);
          }
        }
      }
    }
    if (exact)
      exact_row<D>(ExactRow{P.q, P.k, P.v, P.perm ? P.perm + size_t(tl.b) * P.n : nullptr,
                            P.gate, P.out, orow, size_t(tl.b) * P.n, P.n, P.Hkv, tl.kvh, tl.p0 + t,
                            sig_p, P.left, P.right, P.causal, P.accumulate, P.scale_log2});
  }
  if (issued) {  // an abort can leave this thread's last O MMA in flight
    umma_commit(bars + 8 * (kDrainH + h));
    const long long t0 = clock64();
    while (!mbar_try_wait(bars + 8 * (kDrainH + h), 0) && clock64() - t0 < kDrainCycles) {
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) sa_chunk_kernel(const __grid_constant__ Params P) {
  extern __shared__ uint8_t smem_raw[];
  // Align by pointer arithmetic on the shared array (not through an integer)
  // so the compiler keeps the shared address space.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + P.off_bar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P.off_bar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.off_bar + 8 * kNumBars + 4);
  volatile int* vote = reinterpret_cast<volatile int*>(smem + P.off_bar + 8 * kNumBars + 8);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bars + 8 * (kQfull + s), kProducers);
      mbar_init(bars + 8 * (kQfree + s), 2 + 8);  // one commit per half, one per softmax warp
      mbar_init(bars + 8 * (kCfull + s), kProducers);
      mbar_init(bars + 8 * (kCfree + s), 2);  // one commit per half
      mbar_init(bars + 8 * (kSfull + s), 1);
      mbar_init(bars + 8 * (kPfull + s), 4);
      mbar_init(bars + 8 * (kPVdone + s), 1);
      mbar_init(bars + 8 * (kOfull + s), 1);
      mbar_init(bars + 8 * (kOfree + s), 4);
    }
    mbar_init(bars + 8 * kDrain, 1);
    mbar_init(bars + 8 * (kDrainH + 0), 1);
    mbar_init(bars + 8 * (kDrainH + 1), 1);
    *abort_flag = 0;
    *vote = 1;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
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

  // Each branch ends with its own CTA-wide barrier: no code runs after the
  // branches under two register limits.
  if (warp >= kFirstSoftmaxWarp) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    if (P.causal)
      softmax_role<D, true>(P, smem, sbase, tmem_base, bars, abort_flag);
    else
      softmax_role<D, false>(P, smem, sbase, tmem_base, bars, abort_flag);
    tc_fence_before();
    __syncthreads();
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    if (warp < kMmaWarp) {
      producer_role<D>(P, smem, sbase, bars, abort_flag, vote);
    } else {
      if ((threadIdx.x & 31) == 0) mma_role<D>(P, sbase, tmem_base, bars, abort_flag);
      __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
      tc_fence_after();
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(uint32_t(P.tmem_alloc))
                   : "memory");
    }
  }
}

// ------------------------------------------------------------------ host
struct Config {
  int Bt, log2g, left, right, nchunks, qstages;
  uint32_t q_bytes, kv_bytes, off_k, off_v, off_csig, off_qtok, off_bits, off_bar, smem_bytes;
};

static uint32_t round_up(uint32_t x, uint32_t m) { return (x + m - 1) / m * m; }

static bool make_config(const Problem& pb, Path path, Config& c) {
  if (pb.d != 64 && pb.d != 128) return false;
  if (pb.g < 1 || pb.g > 32 || kBM % pb.g != 0) return false;
  c.Bt = kRows / pb.g;  // tokens of a (256-row) tile
  c.log2g = 0;
  while ((1 << c.log2g) < pb.g) ++c.log2g;
  if (path == kPathSA) {
    c.left = c.right = pb.window / 2;
  } else {
    c.left = pb.window_swa - 1;
    c.right = 0;
  }
  const long long span = (long long)c.Bt + c.left + c.right;
  const long long nch = (span + kKC - 1) / kKC;
  if (nch > (1 << 20)) return false;
  c.nchunks = int(nch);
  c.q_bytes = kBM * pb.d * 2;  // one half of the Q tile
  c.kv_bytes = kKC * pb.d * 2;
  for (c.qstages = 2; c.qstages >= 1; --c.qstages) {  // two Q stages when they fit
    c.off_k = uint32_t(c.qstages) * 2 * c.q_bytes;
    c.off_v = c.off_k + 2 * c.kv_bytes;
    c.off_csig = c.off_v + 2 * c.kv_bytes;
    c.off_qtok = c.off_csig + 2u * kKC * 4;
    c.off_bits = c.off_qtok + uint32_t(c.qstages * kRows) * 4;
    // mask words (8 warps x 2 stages x 32 tokens x 4) and the warps' tokens
    c.off_bar = round_up(c.off_bits + 8u * 2 * 32 * kSub * 4 + 8 * 32 * 4, 64);
    c.smem_bytes = c.off_bar + 8 * kNumBars + 16 + 1024;  // + slot, flags, alignment slack
    if (c.smem_bytes <= kMaxSmem) return true;
  }
  return false;
}

static bool device_sm103(int* sms) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (sms) cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  return major == 10 && minor == 3;
}

template <int D>
static cudaError_t launch_one(int grid, uint32_t smem, cudaStream_t stream, const Params& P) {
  cudaError_t ce = cudaFuncSetAttribute(sa_chunk_kernel<D>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (ce != cudaSuccess) return ce;
  cudaFuncAttributes fa;
  ce = cudaFuncGetAttributes(&fa, sa_chunk_kernel<D>);
  if (ce != cudaSuccess) return ce;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;  // register split
  int resident = 0;
  ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, sa_chunk_kernel<D>, kThreads, smem);
  if (ce != cudaSuccess) return ce;
  if (resident < 1) return cudaErrorInvalidConfiguration;
  sa_chunk_kernel<D><<<grid, kThreads, smem, stream>>>(P);
  return cudaGetLastError();
}

}  // namespace chunk

namespace chunk {
// Whether the variant was compiled to the launch register count its
// setmaxnreg split assumes (checked once per variant).
template <int D>
static bool regs_ok() {
  static int cache = -1;
  if (cache < 0) {
    cudaFuncAttributes fa;
    const cudaError_t ce = cudaFuncGetAttributes(&fa, sa_chunk_kernel<D>);
    cache = (ce == cudaSuccess && fa.numRegs == kLaunchRegs) ? 1 : 0;
  }
  return cache == 1;
}
}  // namespace chunk

bool chunk_supported(const Problem& pb, Path path) {
  if (path != kPathSA && path != kPathSWA) return false;
  if (!chunk::device_sm103(nullptr)) return false;
  chunk::Config c;
  if (!chunk::make_config(pb, path, c)) return false;
  return pb.d == 128 ? chunk::regs_ok<128>() : chunk::regs_ok<64>();
}

sa_status_t launch_chunk(const Problem& pb, Path path, const float* gate, int accumulate,
                         cudaStream_t stream) {
  using namespace chunk;
  int sms = 0;
  if (!device_sm103(&sms)) return fail(SA_ERR_UNSUPPORTED, "device is not sm_103");
  Config c;
  if (!make_config(pb, path, c)) return fail(SA_ERR_UNSUPPORTED, "shape does not fit the chunk kernel");
  Params P;
  std::memset(&P, 0, sizeof(P));
  P.q = static_cast<const __nv_bfloat16*>(pb.q);
  P.k = static_cast<const __nv_bfloat16*>(pb.k);
  P.v = static_cast<const __nv_bfloat16*>(pb.v);
  P.perm = (path == kPathSA) ? pb.perm : nullptr;
  P.gate = gate;
  P.out = static_cast<__nv_bfloat16*>(pb.out);
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
  P.nchunks = c.nchunks;
  P.qstages = c.qstages;
  P.causal = (path == kPathSA) ? pb.causal : 0;
  P.accumulate = accumulate;
  P.scale_log2 = pb.scale * 1.4426950408889634f;
  P.tiles_per_seq = (pb.n + c.Bt - 1) / c.Bt;
  P.num_tiles = P.tiles_per_seq * pb.B * pb.Hkv;
  P.q_bytes = c.q_bytes;
  P.kv_bytes = c.kv_bytes;
  P.off_k = c.off_k;
  P.off_v = c.off_v;
  P.off_csig = c.off_csig;
  P.off_qtok = c.off_qtok;
  P.off_bits = c.off_bits;
  P.off_bar = c.off_bar;
  P.tmem_alloc = 512;  // S of the two halves (128 columns each), then their O
  P.timeout_cycles = wait_limit_cycles();
  const int grid = P.num_tiles < sms ? P.num_tiles : sms;
  const cudaError_t ce = (pb.d == 128) ? launch_one<128>(grid, c.smem_bytes, stream, P)
                                       : launch_one<64>(grid, c.smem_bytes, stream, P);
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "chunk kernel launch: %s", cudaGetErrorString(ce));
  return SA_OK;
}

}  // namespace sa
