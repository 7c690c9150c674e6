// Append accepted draft rows to the KV caches ("Technical Summary: Dustin",
// section 3 "Verification Workflow", step 5: accepted tokens are appended to
// the cache, rejected tokens are discarded).  Two launches: the copy (every
// CTA reads the old seq_len), then the seq_len bump.
#include "common.cuh"
#include "kernels.h"

namespace dustin {

namespace {

__device__ __forceinline__ bool append_ok(const AppendArgs& A, int b, int* L_out, int* n_out) {
  const int L = A.seq_len[b];
  const int n = A.n_accept[b];
  *L_out = L;
  *n_out = n;
  return L >= 0 && L <= A.Lcap && n >= 0 && n <= A.T && L + n <= A.Lcap;
}

// grid (hkv, B, n_layers); 128 threads copy up to T rows of K and V
__global__ void append_copy_kernel(const __grid_constant__ AppendArgs A) {
  pdl_launch_dependents();
  pdl_wait();
  const int g = blockIdx.x, b = blockIdx.y, l = blockIdx.z;
  int L, n;
  if (!append_ok(A, b, &L, &n)) return;
  const AppendLayerDev& Ly = A.layer[l];
  const int vec = A.D / 8;   // 16-byte chunks per row
  for (int idx = threadIdx.x; idx < n * vec * 2; idx += blockDim.x) {
    const int which = idx / (n * vec);   // 0: K, 1: V
    const int rem = idx % (n * vec);
    const int u = rem / vec, c = rem % vec;
    const size_t src_off = ((size_t(b) * A.hkv + g) * A.T + u) * A.D + size_t(c) * 8;
    if (which == 0) {
      uint4* dst = reinterpret_cast<uint4*>(Ly.k + size_t(b) * Ly.ksb + size_t(g) * Ly.ksh +
                                            size_t(L + u) * Ly.ksl + size_t(c) * 8);
      *dst = *reinterpret_cast<const uint4*>(Ly.kb + src_off);
    } else {
      uint4* dst = reinterpret_cast<uint4*>(Ly.v + size_t(b) * Ly.vsb + size_t(g) * Ly.vsh +
                                            size_t(L + u) * Ly.vsl + size_t(c) * 8);
      *dst = *reinterpret_cast<const uint4*>(Ly.vb + src_off);
    }
  }
}

__global__ void append_bump_kernel(const __grid_constant__ AppendArgs A) {
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= A.B) return;
  int L, n;
  if (!append_ok(A, b, &L, &n)) {
    flag_error(A.err, DUSTIN_DEV_APPEND);
    return;
  }
  A.seq_len[b] = L + n;
}

}  // namespace

cudaError_t append_launch(const AppendArgs& a, cudaStream_t stream) {
  cudaError_t e = launch_pdl(append_copy_kernel, dim3(a.hkv, a.B, a.n_layers), dim3(128), 0, stream, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(append_bump_kernel, dim3((a.B + 127) / 128), dim3(128), 0, stream, a);
}

}  // namespace dustin
