// sigma^{-1} on the device ("Core mechanism" step 3 of the Stochastic
// Attention summary; "Theoretical properties": the permutation and its
// inverse are O(n) index operations).
//
// Two launches over all B*n positions:
//   1. scatter  inv[b, perm[b, p]] = p   (out-of-range entries -> RANGE bit)
//   2. verify   inv[b, perm[b, p]] == p  (a lost race means a repeated
//               entry -> DUP bit; a repeated entry in a length-n row also
//               leaves some slot unwritten, which the pigeonhole argument
//               ties back to a DUP or RANGE report)
// Both are coalesced 4-byte streams; the scatter writes are random.
#include "sa_internal.h"

namespace sa {
namespace {

__global__ void inv_scatter_kernel(const int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                                   int n, long long total, int32_t* err) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const long long b = idx / n;
  const int p = int(idx - b * n);
  const int i = perm[idx];
  if (i < 0 || i >= n) {
    atomicOr(err, SA_ERRBIT_RANGE);
    return;
  }
  inv[b * n + i] = p;
}

__global__ void inv_verify_kernel(const int32_t* __restrict__ perm, const int32_t* __restrict__ inv,
                                  int n, long long total, int32_t* err) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const long long b = idx / n;
  const int p = int(idx - b * n);
  const int i = perm[idx];
  if (i < 0 || i >= n) return;  // already reported by the scatter
  if (inv[b * n + i] != p) atomicOr(err, SA_ERRBIT_DUP);
}

}  // namespace

sa_status_t launch_inverse_perm(const int32_t* perm, int32_t* inv, int batch, int n,
                                int32_t* err, cudaStream_t stream) {
  const long long total = (long long)batch * n;
  const int threads = 256;
  const unsigned blocks = unsigned((total + threads - 1) / threads);
  inv_scatter_kernel<<<blocks, threads, 0, stream>>>(perm, inv, n, total, err);
  cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "inverse-perm scatter launch: %s", cudaGetErrorString(ce));
  inv_verify_kernel<<<blocks, threads, 0, stream>>>(perm, inv, n, total, err);
  ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(SA_ERR_CUDA, "inverse-perm verify launch: %s", cudaGetErrorString(ce));
  return SA_OK;
}

}  // namespace sa
