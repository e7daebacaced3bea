// Receptive fields of stacked SA layers on the GPU.
//
// "Theoretical properties", receptive-field bullet of the Stochastic
// Attention summary: with an independent sigma per layer, the set of tokens
// whose information reaches token i grows far faster than sliding-window
// attention's l * w, reaching the whole sequence in O(log_w n) layers.  With
// N_l(i) token i's neighbour set in layer l ("Core mechanism": the tokens at
// permuted positions within h = floor(w/2) of i's position, truncated at the
// ends; causal: also no later than i), the receptive field is
//   R_0(i) = {i},   R_l(i) = union over j in N_l(i) of R_{l-1}(j),
// so R_L(i) = N_1(... N_L({i}) ...): the outermost layer L acts on {i} first.
//
// For a batch of target tokens the kernels carry one bit per target in a
// 64-bit word per token (64 targets per pass).  One layer step maps a set S
// to the union of N_l(j) over j in S:
//   k is in S'  iff  some permuted position q within h of k's position
//                    holds a token j in S (and, when causal, j >= k),
// evaluated per position p with k = sigma_l[p] as an OR over the window of
// the words of sigma_l[q] (with the causal test per key), which handles all
// 64 targets at once.  A popcount per target bit then gives |R_L|.
#include "sa_internal.h"

namespace sa {
namespace graph {

__global__ void rf_seed(unsigned long long* words, const int32_t* targets, int t0, int cnt, int n,
                        int32_t* err) {
  const int t = threadIdx.x;
  if (t < cnt) {
    const int k = targets[t0 + t];
    if (unsigned(k) >= unsigned(n)) {
      atomicOr(err, SA_ERRBIT_RANGE);
      return;
    }
    atomicOr(words + k, 1ull << t);
  }
}

// One layer: dst[sigma[p]] = OR over q in [p-h, p+h] of src[sigma[q]], keys
// restricted to sigma[q] >= sigma[p] when causal.  The block stages its
// positions' window of tokens and words in shared memory.
constexpr int kTile = 1024;
constexpr int kMaxHalf = 1024;

__global__ void __launch_bounds__(kTile) rf_step(const unsigned long long* __restrict__ src,
                                                 unsigned long long* __restrict__ dst,
                                                 const int32_t* __restrict__ perm, int n, int h,
                                                 int causal, int32_t* err) {
  extern __shared__ unsigned long long s_words[];  // [kTile + 2h]
  int32_t* s_tok = reinterpret_cast<int32_t*>(s_words + kTile + 2 * h);
  const int p0 = blockIdx.x * kTile;
  const int span = kTile + 2 * h;
  for (int i = threadIdx.x; i < span; i += blockDim.x) {
    const int q = p0 - h + i;
    int tok = -1;
    unsigned long long w = 0;
    if (q >= 0 && q < n) {
      tok = perm[q];
      if (unsigned(tok) >= unsigned(n)) {
        atomicOr(err, SA_ERRBIT_RANGE);
        tok = -1;
      } else {
        w = src[tok];
      }
    }
    s_tok[i] = tok;
    s_words[i] = w;
  }
  __syncthreads();
  const int p = p0 + threadIdx.x;
  if (p >= n) return;
  const int k = s_tok[threadIdx.x + h];
  if (k < 0) return;
  unsigned long long acc = 0;
  const int lo = threadIdx.x, hi = threadIdx.x + 2 * h;  // window in the staged span
  if (causal) {
    for (int i = lo; i <= hi; ++i)
      if (s_tok[i] >= k) acc |= s_words[i];
  } else {
    for (int i = lo; i <= hi; ++i) acc |= s_words[i];
  }
  dst[k] = acc;
}

// The same layer without the causal test: the window OR of every position
// comes from a doubling table built in shared memory.  Level L holds the OR
// of 2^L consecutive staged words; with 2^L <= 2h+1 < 2^(L+1) a window is
// the OR of two level-L entries (overlapping), so each position costs two
// reads after ~log2(2h+1) passes over the staged span, instead of 2h+1.
__global__ void __launch_bounds__(kTile) rf_step_nc(const unsigned long long* __restrict__ src,
                                                    unsigned long long* __restrict__ dst,
                                                    const int32_t* __restrict__ perm, int n, int h,
                                                    int32_t* err) {
  extern __shared__ unsigned long long s_tab[];  // two [kTile + 2h] tables, then [kTile] tokens
  const int span = kTile + 2 * h;
  unsigned long long* cur = s_tab;
  unsigned long long* nxt = s_tab + span;
  int32_t* s_tok = reinterpret_cast<int32_t*>(s_tab + 2 * span);
  const int p0 = blockIdx.x * kTile;
  for (int i = threadIdx.x; i < span; i += blockDim.x) {
    const int q = p0 - h + i;
    int tok = -1;
    unsigned long long w = 0;
    if (q >= 0 && q < n) {
      tok = perm[q];
      if (unsigned(tok) >= unsigned(n)) {
        atomicOr(err, SA_ERRBIT_RANGE);
        tok = -1;
      } else {
        w = src[tok];
      }
    }
    cur[i] = w;
    if (i >= h && i < h + kTile) s_tok[i - h] = tok;
  }
  __syncthreads();
  const int width = 2 * h + 1;
  int len = 1;
  while (2 * len <= width) {
    // entries past span - 2 len are never read again
    for (int i = threadIdx.x; i + len < span; i += blockDim.x) nxt[i] = cur[i] | cur[i + len];
    __syncthreads();
    unsigned long long* t = cur;
    cur = nxt;
    nxt = t;
    len *= 2;
  }
  const int p = p0 + threadIdx.x;
  if (p >= n) return;
  const int k = s_tok[threadIdx.x];
  if (k < 0) return;
  // window [threadIdx.x, threadIdx.x + width) of the staged span
  dst[k] = cur[threadIdx.x] | cur[threadIdx.x + width - len];
}

// sizes[t0 + t] += number of tokens whose word has bit t set.
__global__ void rf_count(const unsigned long long* __restrict__ words, int n, int cnt,
                         int64_t* __restrict__ sizes_row, int t0) {
  __shared__ unsigned int s_cnt[64];
  if (threadIdx.x < 64) s_cnt[threadIdx.x] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  unsigned int local[2] = {0, 0};  // this lane's two bits: lane and lane + 32
  // warp-uniform loop (the shuffles below need every lane)
  for (int base = blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < n;
       base += gridDim.x * blockDim.x) {
    const int k = base + lane;
    const unsigned long long w = k < n ? words[k] : 0ull;
    // every lane of the warp counts its two bit positions over the warp's 32 words
    for (int src = 0; src < 32; ++src) {
      const unsigned long long ws = __shfl_sync(0xffffffffu, w, src);
      local[0] += unsigned((ws >> lane) & 1ull);
      local[1] += unsigned((ws >> (lane + 32)) & 1ull);
    }
  }
  atomicAdd(&s_cnt[lane], local[0]);
  atomicAdd(&s_cnt[lane + 32], local[1]);
  __syncthreads();
  if (threadIdx.x < cnt) atomicAdd(reinterpret_cast<unsigned long long*>(sizes_row + t0 + threadIdx.x),
                                   (unsigned long long)s_cnt[threadIdx.x]);
}

}  // namespace graph

size_t receptive_field_workspace_bytes(int n) { return 2 * size_t(n) * sizeof(unsigned long long); }

sa_status_t launch_receptive_field(const int32_t* perms, int layers, int n, int window, int causal,
                                   const int32_t* targets, int num_targets, int64_t* sizes,
                                   void* workspace, int32_t* err, cudaStream_t s) {
  using namespace graph;
  const int h = window / 2 < n - 1 ? window / 2 : n - 1;
  if (h > kMaxHalf) return fail(SA_ERR_UNSUPPORTED, "window/2 above %d", kMaxHalf);
  unsigned long long* wa = static_cast<unsigned long long*>(workspace);
  unsigned long long* wb = wa + n;
  const size_t wbytes = size_t(n) * sizeof(unsigned long long);
  cudaError_t ce = cudaMemsetAsync(sizes, 0, size_t(layers) * num_targets * sizeof(int64_t), s);
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "clearing sizes: %s", cudaGetErrorString(ce));
  const int step_blocks = (n + kTile - 1) / kTile;
  const size_t step_smem = causal
      ? size_t(kTile + 2 * h) * (sizeof(unsigned long long) + sizeof(int32_t))
      : size_t(kTile + 2 * h) * 2 * sizeof(unsigned long long) + size_t(kTile) * sizeof(int32_t);
  ce = causal ? cudaFuncSetAttribute(rf_step, cudaFuncAttributeMaxDynamicSharedMemorySize, int(step_smem))
              : cudaFuncSetAttribute(rf_step_nc, cudaFuncAttributeMaxDynamicSharedMemorySize, int(step_smem));
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "rf_step attribute: %s", cudaGetErrorString(ce));
  const int count_blocks = (n + 255) / 256 < 152 * 4 ? (n + 255) / 256 : 152 * 4;
  for (int t0 = 0; t0 < num_targets; t0 += 64) {
    const int cnt = num_targets - t0 < 64 ? num_targets - t0 : 64;
    for (int L = 1; L <= layers; ++L) {
      // R_L of the group: seed {targets}, then layers L, L-1, ..., 1.
      ce = cudaMemsetAsync(wa, 0, wbytes, s);
      if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "clearing words: %s", cudaGetErrorString(ce));
      rf_seed<<<1, 64, 0, s>>>(wa, targets, t0, cnt, n, err);
      unsigned long long* cur = wa;
      unsigned long long* nxt = wb;
      for (int l = L; l >= 1; --l) {
        if (causal)
          rf_step<<<step_blocks, kTile, step_smem, s>>>(cur, nxt, perms + size_t(l - 1) * n, n, h,
                                                       causal, err);
        else
          rf_step_nc<<<step_blocks, kTile, step_smem, s>>>(cur, nxt, perms + size_t(l - 1) * n, n, h,
                                                          err);
        unsigned long long* t = cur;
        cur = nxt;
        nxt = t;
      }
      rf_count<<<count_blocks, 256, 0, s>>>(cur, n, cnt, sizes + size_t(L - 1) * num_targets, t0);
    }
  }
  ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "receptive-field launch: %s", cudaGetErrorString(ce));
  return SA_OK;
}

}  // namespace sa
