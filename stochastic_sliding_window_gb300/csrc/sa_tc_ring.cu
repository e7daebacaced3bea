// tcgen05 kernel for SA / SWA with a sliding K/V ring in shared memory.
//
// Same attention as sa_tc.cu (Stochastic Attention summary, "Core mechanism"
// steps 1-3; causal rule from "Theoretical properties"; SWA from "Problem
// statement"): a tile is Bt = 128/g consecutive permuted positions of one
// (sequence, kv head) pair stacked with the g query heads of that kv head
// (M = 128 rows), attending over the contiguous permuted key span
// [p0 - left, p0 + Bt - 1 + right].
//
// What differs from the gather kernel is how the operands reach the tensor
// cores.  Each CTA takes a CONTIGUOUS run of tiles.  Consecutive tiles of a
// sequence share all but Bt rows of their key span, so K and V live in a
// ring of R = span + 2*Bt rows and each tile fetches only its Bt new rows
// (plus its 128 Q rows); the first tile of a run fetches the whole span.
// Copier warps fetch rows with TMA four-row gathers (tile::gather4: one
// 128-byte column block of four arbitrary rows per copy, swizzled by the
// copy engine), spread over the lanes of five or six warps: the copy engine's
// intake grows with the number of warps issuing, and the copies take no
// load/store-unit slots from the softmax warps.  Q and K of a tile are
// needed only by S = Q K^T, V only by O = P V, so they land on separate
// barriers and are released separately: a Q stage is free once the S MMA
// of the tile two back has completed, the K rows a tile overwrites once
// that of the tile three back has, V rows once its O MMA has.  The sigma
// values of the next tile's new positions are loaded into registers one
// tile ahead.  The key tokens sigma[q] of the ring are kept twice (slots s
// and s + R) so that a tile's span is always a plain contiguous array.
//
// Roles (four warpgroups, 512 threads):
//   warps 0-4   copiers (0-5 for spans of up to 128 keys): sigma of new
//               positions, TMA gathers of Q / K / V rows
//   warps 5-6   maskers (warp 6 alone for spans of up to 128 keys): the
//               tile's mask words (one 32-bit word per token and
//               32-key chunk, from sigma), then the hand-over to the tile's
//               softmax warpgroup
//   warp 7      lane 0 issues S = Q K^T of every tile in order; the warp
//               owns TMEM
//   warps 8-11  softmax, O MMA and epilogue of even tiles (TMEM stage 0)
//   warps 12-15 softmax, O MMA and epilogue of odd tiles  (TMEM stage 1)
// Per tile: S = Q K^T (one or two MMAs when the span wraps the ring) into
// TMEM; each row's window is read from TMEM in 32-column chunks in two passes
// (a reference maximum -- from three chunks on the maximum over every span
// column, returned by the TMEM loads -- then exponentials) and P is written
// back to TMEM as bf16 over its own S columns; one thread of the warpgroup
// then issues O = P V with P taken from TMEM and V used MN-major straight
// from the ring (so no other warp has to notice that P is ready); the
// epilogue scales by 1/rowsum, optionally applies the gate and the previous
// out row, and scatters row sigma[p0+t].  Mask words and copies are thus off
// the softmax warps' path, which is the longest per tile.
// Every wait is bounded (SA_ERRBIT_TIMEOUT); the copiers wait for their last
// copies to land, and each O issuer for its last MMA, before exit.
#include "sa_internal.h"
#include "sa_tc_common.cuh"

#include <cstring>

namespace sa {
namespace ring {

using namespace tcc;

constexpr int kThreads = 512;
// Warps 0-6 split into copiers (sigma of new positions, TMA copies) and
// maskers (mask words, the hand-over to the softmax warpgroup).  The copies
// per tile do not depend on the span, the mask words grow with it: one
// masker warp for spans of up to four 32-key chunks, two beyond (measured
// best at each).
template <int NCH>
struct Split {
  static constexpr int kCopiers = NCH <= 4 ? 192 : 160;
  static constexpr int kMaskers = 224 - kCopiers;
};
constexpr int kMmaWarp = 7;
constexpr int kFirstSoftmaxWarp = 8;
constexpr int kLaunchRegs = 128;
constexpr int kCtrlRegs = 96;
constexpr int kSoftmaxRegs = 160;
static_assert(256 * kCtrlRegs + 256 * kSoftmaxRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
// Spans up to 256 keys: two TMEM stages of S (P over S) and O fit in 512
// columns for d <= 128; shared memory decides the rest.
constexpr int kMaxChunks = 8;
constexpr int kQStages = 2;  // Q buffers; a stage is free once its S MMA is done
constexpr int kVDepth = 3;   // V (and K) rows of tile x overwrite those of tile x - 3
constexpr uint32_t kMaxSmem = 232448;

struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* perm;  // [B, n]; unused when identity
  const float* gate;    // [B, n, Hq] logits or nullptr
  __nv_bfloat16* out;
  int32_t* err;
  int B, n, Hq, Hkv, g, log2g, Bt;
  int left, right, span_pad, R;
  int causal, accumulate, identity;
  float scale_log2;
  int tiles_per_seq, num_tiles;
  int cols_stage, tmem_alloc;  // TMEM stage width; S at 0, P over S, O at span_pad/2
  uint32_t q_bytes, off_k, off_v, off_sig, off_vtok, off_bits, off_bar;
  long long timeout_cycles;
};

// Barrier slots (8 bytes each) after off_bar.  Q families are indexed by
// it % kQStages, V families by it % kVDepth, warpgroup families by it & 1.
enum : uint32_t {
  kFullQK = 0,   // [kQStages] Q stage and new K rows of tile it landed (TMA bytes)
  kQKdone = 3,   // [kQStages] S MMA of tile it done: its Q stage and K rows are free
  kFullV = 6,    // [kVDepth] new V rows of tile it landed (TMA bytes)
  kPVdone = 9,   // [kVDepth] O MMA of tile it done: its V rows are free
  kSready = 12,  // [2] sigma and mask words of tile it ready (per softmax warpgroup)
  kSfree = 14,   // [2] the warpgroup has read the sigma and words of tile it
  kSfull = 16,   // [2] S of tile it in TMEM stage it & 1
  kPfull = 18,   // [2] P of tile it written to TMEM (the warpgroup's 4 warps)
  kOfull = 20,   // [2] O of tile it in TMEM (committed by the warpgroup's issuer)
  kTempty = 22,  // [2] TMEM stage read out by the epilogue
  kDrain = 24,   // final completion of the S MMAs
  kDrainWg = 25, // [2] final completion of the warpgroup's O MMAs
  kSigW = 27,    // [4] sigma of tile it written to the ring (copiers -> maskers)
  kNumBars = 31,
};
static_assert(kFullQK + kQStages <= kQKdone && kQKdone + kQStages <= kFullV, "barrier slots");
static_assert(32 * kMaxChunks <= 2 * Split<kMaxChunks>::kCopiers,
              "a tile's new positions: two per copier thread");

// Tiles of this CTA: a contiguous range, split evenly over the grid.
__device__ __forceinline__ void cta_range(const Params& P, int& begin, int& end) {
  begin = int((long long)blockIdx.x * P.num_tiles / gridDim.x);
  end = int((long long)(blockIdx.x + 1) * P.num_tiles / gridDim.x);
}

// Walks this CTA's tiles in order keeping the ring mapping: a run of one
// sequence maps key position q to ring slot (q - seg_q0) mod R.  The first
// step locates its tile by division; every later step advances by one tile.
struct TileWalk {
  int seq = -1, seg_q0 = 0;
  int b = 0, kvh = 0, p0 = 0, slot_a = 0;
  int ld0 = 0, nld = 0, ld_slot = 0;  // positions the tile loads, slot of the first
  bool new_seg = false;
  __device__ __forceinline__ void step(const Params& P, int tile) {
    if (seq < 0) {
      seq = tile / P.tiles_per_seq;
      p0 = (tile - seq * P.tiles_per_seq) * P.Bt;
      b = seq / P.Hkv;
      kvh = seq - b * P.Hkv;
      new_seg = true;
    } else {
      p0 += P.Bt;
      new_seg = p0 >= P.n;
      if (new_seg) {
        p0 = 0;
        ++seq;
        if (++kvh == P.Hkv) {
          kvh = 0;
          ++b;
        }
      }
    }
    if (new_seg) {  // a new run: the whole span, from slot 0
      seg_q0 = p0 - P.left;
      slot_a = 0;
      ld0 = seg_q0;
      nld = P.span_pad;
      ld_slot = 0;
    } else {  // Bt new positions at the right end of the span
      slot_a += P.Bt;
      if (slot_a >= P.R) slot_a -= P.R;
      ld0 = p0 - P.left + P.span_pad - P.Bt;
      nld = P.Bt;
      ld_slot = slot_a + P.span_pad - P.Bt;
      if (ld_slot >= P.R) ld_slot -= P.R;
    }
  }
  // Locates a tile from scratch (few registers live across tiles; divides).
  // Sets b, kvh, p0, slot_a and new_seg only.
  __device__ __forceinline__ void locate(const Params& P, int tile) {
    const int s = tile / P.tiles_per_seq;
    p0 = (tile - s * P.tiles_per_seq) * P.Bt;
    b = s / P.Hkv;
    kvh = s - b * P.Hkv;
    new_seg = (s != seq);
    if (new_seg) {
      seq = s;
      seg_q0 = p0 - P.left;
    }
    slot_a = (p0 - P.left - seg_q0) % P.R;  // non-negative within a run
  }
  // ring slot of the tile's i-th loaded position (i < nld <= span_pad < R)
  __device__ __forceinline__ int slot_of(const Params& P, int i) const {
    const int sl = ld_slot + i;
    return sl >= P.R ? sl - P.R : sl;
  }
};

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

// 32-byte global store (sm_100 family): one whole sector per thread.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&r)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
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

// Copiers (warps 0-4 or 0-5): per tile, wait for the slots it reuses
// to retire, write sigma of its new positions to the ring, then issue its
// TMA copies.
template <int D, int NCH>
__device__ void copy_role(const Params& P, const CUtensorMap* tq, const CUtensorMap* tk,
                          const CUtensorMap* tv, uint8_t* smem, uint32_t sbase, uint32_t bars,
                          volatile int* abort_flag, volatile int* votes) {
  constexpr int KB = D / 64;  // 128-byte column blocks per row
  constexpr int kCopiers = Split<NCH>::kCopiers;
  const int tid = threadIdx.x;
  // This thread's place in a tile's TMA issue order: consecutive copies go to
  // different warps (a warp issues its lanes' copies one after another).
  const int issue_idx = (tid & 31) * (kCopiers / 32) + (tid >> 5);
  int32_t* sig2 = reinterpret_cast<int32_t*>(smem + P.off_sig);
  int32_t* vtok = reinterpret_cast<int32_t*>(smem + P.off_vtok);  // [2][span_pad] new tokens
  const uint32_t sk = sbase + P.off_k, sv = sbase + P.off_v;
  auto wait = [&](uint32_t bar, uint32_t par) {
    return bounded_wait(bar, par, P.timeout_cycles, P.err, abort_flag);
  };
  // Thread 0 waits for tiles to retire on a [3] family, each tile once and in
  // order (so no wait is ever two phases behind its barrier).
  int qk_seen = -1, pv_seen = -1;
  auto retire = [&](uint32_t fam, int depth, int& seen, int upto) {
    bool ok = true;
    for (int z = seen + 1; z <= upto && ok; ++z)
      ok = wait(bars + 8 * (fam + z % depth), (z / depth) & 1);
    if (ok && upto > seen) seen = upto;
    return ok;
  };
  // Thread 0's verdict, shared with the other copiers.
  auto agree = [&](volatile int* slot, bool ok) {
    if (tid == 0) *slot = ok ? 1 : 0;
    asm volatile("bar.sync 1, %0;" ::"n"(kCopiers) : "memory");
    return *slot != 0;
  };
  // sigma of a tile's new positions (two per thread at most), into registers;
  // unconditional loads of clamped positions, so nothing waits on them here
  auto fetch = [&](const TileWalk& w, int (&pre)[2]) {
    const int q0 = min(max(w.ld0 + tid, 0), P.n - 1);
    const int q1 = min(max(w.ld0 + tid + kCopiers, 0), P.n - 1);
    if (P.identity) {
      pre[0] = q0;
      pre[1] = q1;
    } else {
      const int32_t* perm_b = P.perm + size_t(w.b) * P.n;
      pre[0] = __ldg(perm_b + q0);
      pre[1] = __ldg(perm_b + q1);
    }
  };
  // Tile it: its sigma, then TMA copies of its Q rows, new K rows and new V
  // rows.  Its Q stage belongs to tile it - kQStages, the K and V rows it
  // overwrites to tile it - 3 (a new run: to every tile in flight, and it
  // rewrites the whole sigma ring, which the warpgroups of those tiles must
  // have read: their O MMA being done implies it).
  auto load = [&](int it, const TileWalk& w, int (&pre)[2], int pv_upto) {
    const int s = it % kQStages;
    const uint32_t full_qk = bars + 8 * (kFullQK + s);
    const uint32_t full_v = bars + 8 * (kFullV + it % kVDepth);
    bool ok = true;
    if (tid == 0) {
      ok = retire(kQKdone, kQStages, qk_seen, w.new_seg ? it - 1 : it - kQStages);
      if (ok) ok = retire(kPVdone, kVDepth, pv_seen, w.new_seg ? it - 1 : pv_upto);
    }
    if (!agree(votes, ok)) return false;
    int32_t* vt = vtok + (it & 1) * P.span_pad;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = tid + kCopiers * k;
      if (i < w.nld) {
        int tok = pre[k];
        if (unsigned(tok) >= unsigned(P.n)) {
          atomicOr(P.err, SA_ERRBIT_RANGE);
          tok = 0;
        }
        const int sl = w.slot_of(P, i);
        sig2[sl] = tok;
        sig2[sl + P.R] = tok;
        vt[i] = tok;
      }
    }
    if (tid == 0) {  // the bytes the tile's copies will deliver, before any is issued
      const uint32_t kv_bytes = uint32_t(w.nld) * D * 2;
      mbar_arrive_expect_tx(full_qk, P.q_bytes + kv_bytes);
      mbar_arrive_expect_tx(full_v, kv_bytes);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kCopiers) : "memory");
    if (tid == 0) mbar_arrive(bars + 8 * (kSigW + (it & 3)));  // sigma visible to the maskers
    // Each copy is a 4-row gather of one 128-byte column block, landing as
    // 512 contiguous swizzled bytes: Q rows r = t*g + j (4 per copy), then the
    // new K rows, then the new V rows (4 ring slots per copy; ring slots and
    // counts are multiples of 4, so a group never wraps).
    const int nq = (kBM / 4) * KB, nk = (w.nld / 4) * KB;
    const int total = nq + 2 * nk;
    const uint32_t sq = sbase + uint32_t(s) * P.q_bytes;
    const int32_t* sig_win = sig2 + w.slot_a + P.left;
    const int rowbase = w.b * P.n;
    for (int i = issue_idx; i < total; i += kCopiers) {
      int rows[4];
      if (i < nq) {
        const int rg = i / KB, kb = i - rg * KB;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = 4 * rg + e;
          rows[e] = (rowbase + sig_win[r >> P.log2g]) * P.Hq + w.kvh * P.g + (r & (P.g - 1));
        }
        tma_gather4(sq + kb * (kBM * 128) + rg * 512, tq, kb * 64, rows[0], rows[1], rows[2],
                    rows[3], full_qk);
      } else {
        const bool is_v = i >= nq + nk;
        const int x = i - nq - (is_v ? nk : 0);
        const int gi = x / KB, kb = x - gi * KB;
#pragma unroll
        for (int e = 0; e < 4; ++e) rows[e] = (rowbase + vt[4 * gi + e]) * P.Hkv + w.kvh;
        const uint32_t dst = kb * (P.R * 128) + w.slot_of(P, 4 * gi) * 128;
        tma_gather4((is_v ? sv : sk) + dst, is_v ? tv : tk, kb * 64, rows[0], rows[1], rows[2],
                    rows[3], is_v ? full_v : full_qk);
      }
    }
    return true;
  };

  int begin, end;
  cta_range(P, begin, end);
  const int ntiles = end - begin;
  TileWalk cur, nxt;
  int pre[2] = {0, 0};
  if (ntiles > 0) {
    nxt.step(P, begin);
    fetch(nxt, pre);
  }
  // V rows of tile x overwrite those of tile x - 3 (a new run: of every tile
  // in flight); the wait is folded into the tile's first wait.
  int issued = 0;
  for (int it = 0; it < ntiles; ++it) {
    cur = nxt;
    const int pv_upto = cur.new_seg ? it - 1 : it - kVDepth;
    const bool ok = load(it, cur, pre, pv_upto);
    if (!ok) break;
    issued = it + 1;
    if (it + 1 < ntiles) {
      nxt.step(P, 0);
      fetch(nxt, pre);
    }
  }
  // The copies of the last tiles land before the CTA may exit (each barrier
  // below was last armed by the tile waited for, so no wait is ambiguous).
  if (tid == 0 && issued > 0) {
    const int last = issued - 1;
    auto drain = [&](uint32_t bar, uint32_t par) {
      const long long t0 = clock64();
      while (!mbar_try_wait(bar, par) && clock64() - t0 < kDrainCycles) {
      }
    };
    for (int x = max(0, last - kQStages + 1); x <= last; ++x)
      drain(bars + 8 * (kFullQK + x % kQStages), (x / kQStages) & 1);
    for (int x = max(0, last - kVDepth + 1); x <= last; ++x)
      drain(bars + 8 * (kFullV + x % kVDepth), (x / kVDepth) & 1);
  }
}

// Maskers (the other warps up to 6): per tile, once its sigma is in the
// ring, the mask words, one per (token, 32-key chunk): bit e set iff key
// column ch*32 + e lies in the token's window (truncated at the sequence
// ends) and, when causal, sigma[q] <= sigma[p]; then hand the tile to its
// softmax warpgroup.  Four word buffers, so that a warpgroup still reading
// the words of tile it - 2 is never overwritten.
template <int NCH>
__device__ void mask_role(const Params& P, uint8_t* smem, uint32_t bars, volatile int* abort_flag,
                          volatile int* votes) {
  constexpr int kMaskers = Split<NCH>::kMaskers;
  const int mt = threadIdx.x - Split<NCH>::kCopiers;  // 0 .. kMaskers - 1
  const int lane = mt & 31, mw = mt >> 5;
  const int32_t* sig2 = reinterpret_cast<const int32_t*>(smem + P.off_sig);
  auto wait = [&](uint32_t bar, uint32_t par) {
    return bounded_wait(bar, par, P.timeout_cycles, P.err, abort_flag);
  };
  int begin, end;
  cta_range(P, begin, end);
  const int ntiles = end - begin;
  TileWalk w;
  for (int it = 0; it < ntiles; ++it) {
    w.step(P, begin + it);
    bool ok = true;
    if (mt == 0) ok = wait(bars + 8 * (kSigW + (it & 3)), (it >> 2) & 1);
    if (mt == 0) votes[2] = ok ? 1 : 0;
    asm volatile("bar.sync 2, %0;" ::"n"(kMaskers) : "memory");
    if (!votes[2]) break;
    const int32_t* sig = sig2 + w.slot_a;
    uint32_t* wbuf = reinterpret_cast<uint32_t*>(smem + P.off_bits) +
                     ((it & 1) * 2 + ((it >> 1) & 1)) * (P.Bt * NCH);
    const int nblk = (P.Bt + 31) >> 5;
    for (int item = mw; item < nblk * NCH; item += kMaskers / 32) {
      const int tb = item / NCH, ch = item - tb * NCH;
      const int tt = tb * 32 + lane;
      const int lo = max(tt, P.left - w.p0);
      const int hi = w.p0 + tt < P.n ? min(tt + P.left + P.right, P.n - 1 - w.p0 + P.left) : -1;
      uint32_t word = band_bits(lo, hi, ch * 32);
      if (P.causal) {
        // lane tt compares its token's sigma with the chunk's 32 key tokens,
        // read four at a time by all lanes together (broadcast loads)
        const int st = sig[P.left + min(tt, P.Bt - 1)];
        const int4* s4p = reinterpret_cast<const int4*>(sig + ch * 32);
        uint32_t cw = 0u;
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const int4 s4 = s4p[e4];
          cw |= (s4.x <= st ? 1u : 0u) << (4 * e4);
          cw |= (s4.y <= st ? 1u : 0u) << (4 * e4 + 1);
          cw |= (s4.z <= st ? 1u : 0u) << (4 * e4 + 2);
          cw |= (s4.w <= st ? 1u : 0u) << (4 * e4 + 3);
        }
        word &= cw;
      }
      if (tt < P.Bt) wbuf[tt * NCH + ch] = word;
    }
    asm volatile("bar.sync 2, %0;" ::"n"(kMaskers) : "memory");
    if (mt == 0) {
      // Hand the tile to its softmax warpgroup once the warpgroup has read
      // what it needed from its previous tile (so this barrier is never two
      // phases ahead of its waiter).
      // A wait that gives up sets the abort flag, which ends every role's
      // next wait (the maskers leave at the top of their next tile together).
      const int wg = it & 1;
      if (wait(bars + 8 * (kSfree + wg), ((it >> 1) & 1) ^ 1)) mbar_arrive(bars + 8 * (kSready + wg));
    }
  }
}

template <int D>
__device__ void mma_role(const Params& P, uint32_t sbase, uint32_t tmem_base, uint32_t bars,
                         volatile int* abort_flag) {
  int begin, end;
  cta_range(P, begin, end);
  const uint32_t ka = sbase + P.off_k;
  auto qk = [&](int it, int slot_a) {
    const int s = it % kQStages, ts = it & 1;
    tc_fence_after();
    const uint32_t d = tmem_base + uint32_t(ts * P.cols_stage);
    const uint32_t qa = sbase + uint32_t(s) * P.q_bytes;
    const int n1 = min(P.span_pad, P.R - slot_a);
    const int n2 = P.span_pad - n1;
    // Descriptors of the first K step; later steps add their byte offset / 16
    // to the start-address field (every operand lies below 256 KB, so the
    // field never carries).
    const uint64_t a0 = sdesc_sw128(qa, 16, 1024);
    const uint64_t b0 = sdesc_sw128(ka + slot_a * 128, 16, 1024);
    const uint64_t w0 = sdesc_sw128(ka, 16, 1024);  // the part past the ring's end
    const uint64_t ring_blk = uint64_t(P.R) * 8;   // next 64-column block of the ring
    const uint32_t id1 = idesc_bf16(kBM, n1, 0), id2 = idesc_bf16(kBM, n2, 0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint64_t da = uint64_t((kk >> 2) * (kBM * 128 / 16) + (kk & 3) * 2);
      const uint64_t db = uint64_t(kk >> 2) * ring_blk + uint64_t((kk & 3) * 2);
      umma_bf16(d, a0 + da, b0 + db, id1, kk > 0 ? 1u : 0u);
      if (n2 > 0) umma_bf16(d + n1, a0 + da, w0 + db, id2, kk > 0 ? 1u : 0u);
    }
    umma_commit(bars + 8 * (kSfull + ts));
    umma_commit(bars + 8 * (kQKdone + s));
  };
  // S = Q K^T of every tile in order, each once its Q and K rows have landed
  // and its TMEM stage has been read out by the epilogue of the tile two
  // back.  (The O MMAs are issued by the softmax warpgroups themselves.)
  const int ntiles = end - begin;
  TileWalk tq;
  for (int it = 0; it < ntiles; ++it) {
    if (!bounded_wait(bars + 8 * (kFullQK + it % kQStages), (it / kQStages) & 1, P.timeout_cycles,
                      P.err, abort_flag))
      break;
    if (!bounded_wait(bars + 8 * (kTempty + (it & 1)), ((it >> 1) & 1) ^ 1, P.timeout_cycles, P.err,
                      abort_flag))
      break;
    tq.step(P, begin + it);
    qk(it, tq.slot_a);
  }
  umma_commit(bars + 8 * kDrain);
  const long long t0 = clock64();
  while (!mbar_try_wait(bars + 8 * kDrain, 0) && clock64() - t0 < kDrainCycles) {
  }
}

// The row's mask word of 32-column chunk ch (the words are in registers; a
// select chain, not a local-memory index).
template <int NCH>
__device__ __forceinline__ uint32_t word_of(const uint32_t (&wd)[NCH], int ch) {
  uint32_t b = wd[0];
#pragma unroll
  for (int k = 1; k < NCH; ++k) b = ch == k ? wd[k] : b;
  return b;
}

template <int D, int NCH, bool kCausal>
__device__ void softmax_role(const Params& P, uint8_t* smem, uint32_t sbase, uint32_t tmem_base,
                             uint32_t bars, volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = (warp - kFirstSoftmaxWarp) >> 2;  // also this warpgroup's TMEM stage
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const int t = r >> P.log2g;
  const int j = r & (P.g - 1);
  const int32_t* sig2 = reinterpret_cast<const int32_t*>(smem + P.off_sig);
  const uint32_t trow = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(wg * P.cols_stage);
  const uint32_t o_col = uint32_t(P.span_pad / 2);
  const bool issuer = quad == 0 && lane == 0;  // issues this warpgroup's O MMAs
  bool issued = false;
  auto wwait = [&](uint32_t bar, uint32_t par) {
    const bool ok = bounded_wait(bar, par, P.timeout_cycles, P.err, abort_flag);
    return __all_sync(0xffffffffu, ok);
  };
  int begin, end;
  cta_range(P, begin, end);
  TileWalk tw;
  int it = 0;
  for (int tile = begin; tile < end; ++tile, ++it) {
    tw.locate(P, tile);
    if ((it & 1) != wg) continue;
    const uint32_t ph = uint32_t(it >> 1) & 1u;
    if (!wwait(bars + 8 * (kSready + wg), ph)) break;  // sigma of the tile is visible
    const int32_t* sig = sig2 + tw.slot_a;            // sigma of span column c is sig[c]
    bool row_valid = tw.p0 + t < P.n;
    const int sig_p = sig[P.left + t];
    // the row's mask words (written by the maskers)
    const uint32_t* wrow = reinterpret_cast<const uint32_t*>(smem + P.off_bits) +
                           (wg * 2 + ((it >> 1) & 1)) * (P.Bt * NCH) + t * NCH;
    uint32_t wd[NCH];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) wd[ch] = wrow[ch];
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (kSfree + wg));  // sigma and words no longer read
    if (row_valid && unsigned(sig_p) >= unsigned(P.n)) {  // never expected: record, skip
      atomicOr(P.err, SA_ERRBIT_INTERNAL);
      row_valid = false;
    }

    if (!wwait(bars + 8 * (kSfull + wg), ph)) break;
    tc_fence_after();
    // Two passes over the row's 32-column chunks, loops kept rolled so the
    // code stays small (the roles share each SM's instruction cache):
    // a reference maximum, then p = 2^(s*scale*log2e - reference) for
    // attended columns (0 elsewhere) written back to TMEM as bf16 over the
    // row's own S columns (P column pair c/2 holds keys c and c+1; chunk ch's
    // P lands on S columns already consumed).
    // From three chunks on, the reference is the maximum over ALL the span's
    // columns, attended or not, which the TMEM loads return themselves (no
    // mask test, no compare per element).  Every span column is a real key
    // of this launch (a position past either end loads a clamped token's
    // row), so for finite inputs the reference is finite and at least the
    // attended maximum: no p exceeds 1.  Softmax does not depend on the
    // reference; a reference so far above the attended maximum that the
    // attended p underflow shows as a row sum below 2^-60, and that row is
    // recomputed exactly (exact_row).  Spans of one or two chunks keep the
    // attended maximum, which costs no more there.
    float mx = -INFINITY;
    if constexpr (NCH <= 2) {
#pragma unroll 1
      for (int ch = 0; ch < NCH; ++ch) {
        uint32_t v[32];
        tmem_ld32(trow + ch * 32, v);
        const uint32_t bits = word_of(wd, ch);
        float m0 = mx, m1 = -INFINITY;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float x0 = (bits >> e) & 1u ? __uint_as_float(v[e]) : -INFINITY;
          const float x1 = (bits >> (e + 1)) & 1u ? __uint_as_float(v[e + 1]) : -INFINITY;
          const float x2 = (bits >> (e + 2)) & 1u ? __uint_as_float(v[e + 2]) : -INFINITY;
          const float x3 = (bits >> (e + 3)) & 1u ? __uint_as_float(v[e + 3]) : -INFINITY;
          m0 = fmax3(m0, x0, x1);
          m1 = fmax3(m1, x2, x3);
        }
        mx = fmaxf(m0, m1);
      }
    } else {
#pragma unroll 1
      for (int ch = 0; ch < NCH; ++ch) mx = fmaxf(mx, tmem_max32(trow + ch * 32));
    }
    const float ms = (mx == -INFINITY) ? 0.f : mx * P.scale_log2;
    const uint64_t sl2 = f2_pack(P.scale_log2, P.scale_log2);
    const uint64_t nms = f2_pack(-ms, -ms);
    uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll 1
    for (int ch = 0; ch < NCH; ++ch) {
      uint32_t v[32];
      tmem_ld32(trow + ch * 32, v);
      const uint32_t bits = word_of(wd, ch);
      uint32_t pk[16];
#pragma unroll
      for (int e2 = 0; e2 < 16; ++e2) {
        const float2 x = f2_unpack(f2_fma(f2_pack(__uint_as_float(v[2 * e2]),
                                                  __uint_as_float(v[2 * e2 + 1])),
                                          sl2, nms));
        const float p0 = (bits >> (2 * e2)) & 1u ? fast_exp2(x.x) : 0.f;
        const float p1 = (bits >> (2 * e2 + 1)) & 1u ? fast_exp2(x.y) : 0.f;
        acc2[e2 & 1] = f2_add(acc2[e2 & 1], f2_pack(p0, p1));
        pk[e2] = pack_bf16x2(p0, p1);
      }
      tmem_st16(trow + ch * 16, pk);
    }
    const float2 a01 = f2_unpack(acc2[0]), a23 = f2_unpack(acc2[1]);
    const float l = (a01.x + a01.y) + (a23.x + a23.y);
    // l is at least the row's largest attended p, 2^-(reference - attended
    // maximum) (every valid row attends its own key): l < 2^-60 means that
    // gap is above 60
    const bool exact = row_valid && l < 0x1p-60f;
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (kPfull + wg));
    // Once P of all 128 rows is in TMEM and the tile's V rows have landed,
    // one thread of the warpgroup issues O = P V (A = P from this stage, B =
    // V straight from the ring, MN-major).  The span's older V rows came with
    // earlier tiles, whose copies complete on their own barriers in any
    // order: waiting for the previous tile's O MMA (which waited for its own
    // rows and, in turn, for the O MMA before it) covers them all.  The other
    // warpgroup issues that MMA, and this thread issued the one two tiles
    // back, so the phase waited for is never two behind or ahead.  Every
    // wait is bounded like every other wait.
    if (issuer &&
        bounded_wait(bars + 8 * (kPfull + wg), ph, P.timeout_cycles, P.err, abort_flag) &&
        bounded_wait(bars + 8 * (kFullV + it % kVDepth), (it / kVDepth) & 1, P.timeout_cycles,
                     P.err, abort_flag) &&
        (it == 0 || bounded_wait(bars + 8 * (kPVdone + (it - 1) % kVDepth),
                                 ((it - 1) / kVDepth) & 1, P.timeout_cycles, P.err, abort_flag))) {
      tc_fence_after();
      const uint32_t stage = tmem_base + uint32_t(wg * P.cols_stage);
      const uint32_t idesc_pv = idesc_bf16(kBM, D, 1);
      const int ksteps = P.span_pad / 16;
      int vs = tw.slot_a;
      uint64_t bd = sdesc_sw128(sbase + P.off_v + vs * 128, P.R * 128, 1024);
      const uint64_t wrap = uint64_t(P.R) * 8;  // R rows of 128 B, in 16-byte units
      for (int kk = 0; kk < ksteps; ++kk) {
        umma_bf16_ts(stage + o_col, stage + 8 * kk, bd, idesc_pv, kk > 0 ? 1u : 0u);
        vs += 16;
        bd += 128;  // 16 rows of 128 B
        if (vs >= P.R) {
          vs -= P.R;
          bd -= wrap;
        }
      }
      umma_commit(bars + 8 * (kOfull + wg));
      umma_commit(bars + 8 * (kPVdone + it % kVDepth));
      issued = true;
    }

    // epilogue
    if (!wwait(bars + 8 * (kOfull + wg), ph)) break;
    tc_fence_after();
    float mul = l > 0.f ? 1.f / l : 0.f;
    const size_t orow =
        row_valid ? (size_t(tw.b) * P.n + sig_p) * P.Hq + size_t(tw.kvh) * P.g + j : 0;
    if (P.gate != nullptr && row_valid) mul *= 1.f / (1.f + expf(-P.gate[orow]));
    // O leaves TMEM in 64-column halves (fewer registers held at once); the
    // stage is handed back once the last half is read.
    const uint64_t mul2 = f2_pack(mul, mul);
    __nv_bfloat16* op = P.out + orow * D;
    const bool stores = row_valid && !exact;  // an exact row is written by exact_row
#pragma unroll 1
    for (int hf = 0; hf < D / 64; ++hf) {
      uint32_t o[2][32];
      tmem_ld32_async(trow + o_col + hf * 64, o[0]);
      tmem_ld32_async(trow + o_col + hf * 64 + 32, o[1]);
      tmem_wait_ld();
      reg_fence(o[0]);
      reg_fence(o[1]);
      if (hf == D / 64 - 1) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (kTempty + wg));
      }
      if (stores && !P.accumulate) {
        // Each thread writes its own row, whole 32-byte sectors per store.
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int k = half * 16 + 2 * e;
              const float2 y = f2_unpack(f2_mul(f2_pack(__uint_as_float(o[ch][k]),
                                                        __uint_as_float(o[ch][k + 1])),
                                                mul2));
              pk[e] = pack_bf16x2(y.x, y.y);
            }
            st_global_v8(op + hf * 64 + ch * 32 + half * 16, pk);
          }
        }
      } else if (stores) {
        // Second pass of the gated sum: each thread reads its own row, adds in
        // fp32 and writes it back.
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint4* dst = reinterpret_cast<uint4*>(op + hf * 64 + ch * 32);
          uint4 prev[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) prev[q4] = dst[q4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 y = f2_unpack(f2_mul(f2_pack(__uint_as_float(o[ch][q4 * 8 + 2 * e]),
                                                        __uint_as_float(o[ch][q4 * 8 + 2 * e + 1])),
                                                mul2));
              f[2 * e] = y.x;
              f[2 * e + 1] = y.y;
            }
            const __nv_bfloat162* pv2 = reinterpret_cast<const __nv_bfloat162*>(&prev[q4]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 pf = __bfloat1622float2(pv2[e]);
              f[2 * e] += pf.x;
              f[2 * e + 1] += pf.y;
            }
            dst[q4] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                 pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
          }
        }
      }
    }
    if (exact)
      exact_row<D>(ExactRow{P.q, P.k, P.v, P.identity ? nullptr : P.perm + size_t(tw.b) * P.n,
                            P.gate, P.out, orow, size_t(tw.b) * P.n, P.n, P.Hkv, tw.kvh, tw.p0 + t,
                            sig_p, P.left, P.right, P.causal, P.accumulate, P.scale_log2});
  }
  if (issued) {  // an abort can leave this thread's last O MMA in flight
    umma_commit(bars + 8 * (kDrainWg + wg));
    const long long t0 = clock64();
    while (!mbar_try_wait(bars + 8 * (kDrainWg + wg), 0) && clock64() - t0 < kDrainCycles) {
    }
  }
}

template <int D, int NCH>
__global__ void __launch_bounds__(kThreads, 1)
    sa_ring_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ Params P) {
  extern __shared__ uint8_t smem_raw[];
  // Align by pointer arithmetic on the shared array (not through an integer)
  // so the compiler keeps the shared address space: ld/st.shared, not generic.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + P.off_bar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P.off_bar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.off_bar + 8 * kNumBars + 4);
  volatile int* votes = reinterpret_cast<volatile int*>(smem + P.off_bar + 8 * kNumBars + 8);  // [3]
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(bars + 8 * (kFullQK + s), 1);
      mbar_init(bars + 8 * (kQKdone + s), 1);
    }
    for (int s = 0; s < kVDepth; ++s) {
      mbar_init(bars + 8 * (kFullV + s), 1);
      mbar_init(bars + 8 * (kPVdone + s), 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(bars + 8 * (kSready + w), 1);
      mbar_init(bars + 8 * (kSfree + w), 4);
      mbar_init(bars + 8 * (kSfull + w), 1);
      mbar_init(bars + 8 * (kPfull + w), 4);
      mbar_init(bars + 8 * (kDrainWg + w), 1);
      mbar_init(bars + 8 * (kOfull + w), 1);
      mbar_init(bars + 8 * (kTempty + w), 4);
    }
    mbar_init(bars + 8 * kDrain, 1);
    for (int x = 0; x < 4; ++x) mbar_init(bars + 8 * (kSigW + x), 1);
    *abort_flag = 0;
    votes[0] = 1;
    votes[1] = 1;
    votes[2] = 1;
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
      softmax_role<D, NCH, true>(P, smem, sbase, tmem_base, bars, abort_flag);
    else
      softmax_role<D, NCH, false>(P, smem, sbase, tmem_base, bars, abort_flag);
    tc_fence_before();
    __syncthreads();
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    if (warp < Split<NCH>::kCopiers / 32) {
      copy_role<D, NCH>(P, &tm_q, &tm_k, &tm_v, smem, sbase, bars, abort_flag, votes);
    } else if (warp < kMmaWarp) {
      mask_role<NCH>(P, smem, bars, abort_flag, votes);
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
  int Bt, log2g, left, right, span_pad, R, cols_stage, tmem_alloc;
  uint32_t q_bytes, off_k, off_v, off_sig, off_vtok, off_bits, off_bar, smem_bytes;
};

static uint32_t round_up(uint32_t x, uint32_t m) { return (x + m - 1) / m * m; }

static bool make_config(const Problem& pb, Path path, Config& c) {
  if (pb.d != 64 && pb.d != 128) return false;
  if (kBM % pb.g != 0) return false;
  c.Bt = kBM / pb.g;
  if (c.Bt % 16 != 0) return false;  // ring offsets must be whole 16-row MMA steps
  c.log2g = 0;
  while ((1 << c.log2g) < pb.g) ++c.log2g;
  if (path == kPathSA) {
    c.left = c.right = pb.window / 2;
  } else {
    c.left = pb.window_swa - 1;
    c.right = 0;
  }
  const long long span = (long long)c.Bt + c.left + c.right;
  if (span > 32LL * kMaxChunks) return false;
  c.span_pad = int(round_up(uint32_t(span), 32));
  c.R = int(round_up(uint32_t(c.span_pad + 2 * c.Bt), 16));
  // TMEM stage: S [0, span_pad); P (bf16 pairs) over S [0, span_pad/2);
  // O [span_pad/2, span_pad/2 + d).
  const int width = c.span_pad > c.span_pad / 2 + pb.d ? c.span_pad : c.span_pad / 2 + pb.d;
  c.cols_stage = int(round_up(uint32_t(width), 32));
  uint32_t alloc = 32;
  while (alloc < uint32_t(2 * c.cols_stage)) alloc <<= 1;
  if (alloc > 512) return false;
  c.tmem_alloc = int(alloc);
  c.q_bytes = kBM * pb.d * 2;
  const uint32_t ring_bytes = uint32_t(c.R) * pb.d * 2;
  c.off_k = kQStages * c.q_bytes;
  c.off_v = c.off_k + ring_bytes;
  c.off_sig = c.off_v + ring_bytes;
  c.off_vtok = round_up(c.off_sig + 2u * c.R * 4, 16);
  c.off_bits = round_up(c.off_vtok + 2u * c.span_pad * 4, 16);
  c.off_bar = round_up(c.off_bits + 4u * c.Bt * (c.span_pad / 32) * 4, 64);
  c.smem_bytes = c.off_bar + 8 * kNumBars + 32 + 1024;  // + slot, flags, alignment slack
  return c.smem_bytes <= kMaxSmem;
}

static bool device_sm103(int* sms) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (sms) cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  return major == 10 && minor == 3;
}

struct Maps {
  CUtensorMap q, k, v;
};

template <int D, int NCH>
static cudaError_t launch_one(int grid, uint32_t smem, cudaStream_t stream, const Maps& m,
                              const Params& P) {
  cudaError_t ce = cudaFuncSetAttribute(sa_ring_kernel<D, NCH>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (ce != cudaSuccess) return ce;
  cudaFuncAttributes fa;
  ce = cudaFuncGetAttributes(&fa, sa_ring_kernel<D, NCH>);
  if (ce != cudaSuccess) return ce;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;  // register split
  int resident = 0;
  ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, sa_ring_kernel<D, NCH>, kThreads,
                                                     smem);
  if (ce != cudaSuccess) return ce;
  if (resident < 1) return cudaErrorInvalidConfiguration;
  sa_ring_kernel<D, NCH><<<grid, kThreads, smem, stream>>>(m.q, m.k, m.v, P);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_variant(int nch, int grid, uint32_t smem, cudaStream_t stream,
                                  const Maps& m, const Params& P) {
  switch (nch) {
    case 1: return launch_one<D, 1>(grid, smem, stream, m, P);
    case 2: return launch_one<D, 2>(grid, smem, stream, m, P);
    case 3: return launch_one<D, 3>(grid, smem, stream, m, P);
    case 4: return launch_one<D, 4>(grid, smem, stream, m, P);
    case 5: return launch_one<D, 5>(grid, smem, stream, m, P);
    case 6: return launch_one<D, 6>(grid, smem, stream, m, P);
    case 7: return launch_one<D, 7>(grid, smem, stream, m, P);
    default: return launch_one<D, 8>(grid, smem, stream, m, P);
  }
}

// Whether the variant a shape launches was compiled to exactly the launch
// register count its setmaxnreg split assumes (checked once per variant), so
// that the automatic kernel choice never picks a kernel that would refuse to
// launch.
static_assert(kMaxChunks == 8, "the variant switches list NCH = 1..8");
template <int D>
static bool regs_ok(int nch) {
  static int cache[kMaxChunks + 1] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};
  const int i = nch < 1 ? 1 : (nch > kMaxChunks ? kMaxChunks : nch);
  if (cache[i] < 0) {
    cudaFuncAttributes fa;
    cudaError_t ce;
    switch (i) {
      case 1: ce = cudaFuncGetAttributes(&fa, sa_ring_kernel<D, 1>); break;
      case 2: ce = cudaFuncGetAttributes(&fa, sa_ring_kernel<D, 2>); break;
      case 3: ce = cudaFuncGetAttributes(&fa, sa_ring_kernel<D, 3>); break;
      case 4: ce = cudaFuncGetAttributes(&fa, sa_ring_kernel<D, 4>); break;
      case 5: ce = cudaFuncGetAttributes(&fa, sa_ring_kernel<D, 5>); break;
      case 6: ce = cudaFuncGetAttributes(&fa, sa_ring_kernel<D, 6>); break;
      case 7: ce = cudaFuncGetAttributes(&fa, sa_ring_kernel<D, 7>); break;
      default: ce = cudaFuncGetAttributes(&fa, sa_ring_kernel<D, 8>); break;
    }
    cache[i] = (ce == cudaSuccess && fa.numRegs == kLaunchRegs) ? 1 : 0;
  }
  return cache[i] == 1;
}

}  // namespace ring

bool ring_supported(const Problem& pb, Path path) {
  if (path != kPathSA && path != kPathSWA) return false;
  if (!ring::device_sm103(nullptr)) return false;
  ring::Config c;
  if (!ring::make_config(pb, path, c)) return false;
  const int nch = c.span_pad / 32;
  return pb.d == 128 ? ring::regs_ok<128>(nch) : ring::regs_ok<64>(nch);
}

sa_status_t launch_ring(const Problem& pb, Path path, const float* gate, int accumulate,
                        cudaStream_t stream) {
  using namespace ring;
  int sms = 0;
  if (!device_sm103(&sms)) return fail(SA_ERR_UNSUPPORTED, "device is not sm_103");
  Config c;
  if (!make_config(pb, path, c)) return fail(SA_ERR_UNSUPPORTED, "shape does not fit the ring kernel");
  Params P;
  std::memset(&P, 0, sizeof(P));
  P.q = static_cast<const __nv_bfloat16*>(pb.q);
  P.k = static_cast<const __nv_bfloat16*>(pb.k);
  P.v = static_cast<const __nv_bfloat16*>(pb.v);
  P.perm = pb.perm;
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
  P.span_pad = c.span_pad;
  P.R = c.R;
  P.causal = (path == kPathSA) ? pb.causal : 0;
  P.accumulate = accumulate;
  P.identity = (path == kPathSWA) ? 1 : 0;
  P.scale_log2 = pb.scale * 1.4426950408889634f;
  P.tiles_per_seq = (pb.n + c.Bt - 1) / c.Bt;
  P.num_tiles = P.tiles_per_seq * pb.B * pb.Hkv;
  P.cols_stage = c.cols_stage;
  P.tmem_alloc = c.tmem_alloc;
  P.q_bytes = c.q_bytes;
  P.off_k = c.off_k;
  P.off_v = c.off_v;
  P.off_sig = c.off_sig;
  P.off_vtok = c.off_vtok;
  P.off_bits = c.off_bits;
  P.off_bar = c.off_bar;
  P.timeout_cycles = wait_limit_cycles();
  // Row maps of Q [B*n*Hq, d] and K, V [B*n*Hkv, d]: the copiers gather
  // four arbitrary rows per copy.
  Maps m;
  const uint64_t qrows = uint64_t(pb.B) * pb.n * pb.Hq, kvrows = uint64_t(pb.B) * pb.n * pb.Hkv;
  if (!encode_row_map(&m.q, pb.q, qrows, pb.d, 1) || !encode_row_map(&m.k, pb.k, kvrows, pb.d, 1) ||
      !encode_row_map(&m.v, pb.v, kvrows, pb.d, 1))
    return fail(SA_ERR_CUDA, "ring kernel: tensor map encoding failed");
  const int grid = P.num_tiles < sms ? P.num_tiles : sms;
  const int nch = c.span_pad / 32;
  const cudaError_t ce = (pb.d == 128) ? launch_variant<128>(nch, grid, c.smem_bytes, stream, m, P)
                                       : launch_variant<64>(nch, grid, c.smem_bytes, stream, m, P);
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "ring kernel launch: %s", cudaGetErrorString(ce));
  return SA_OK;
}

}  // namespace sa
