// The literal "compressed target KV cache" ("Technical Summary: Dustin",
// section 3 "Verification Workflow", step 3): the rows of I_verify are copied,
// per layer and KV head, into compact caches of k rows, so that several
// verification passes can read them densely.
//
// One CTA per (run of kRows selected rows, KV head, sequence, layer), so that
// even a small batch spreads over every SM; 16-byte loads and stores, eight
// in flight per thread.  Row j of the compact caches is row i_verify[b][j] of
// the full caches; entries -1 (padding) and invalid indices give zero rows
// (invalid ones are flagged).  The first CTA of layer 0, head 0 of each
// sequence also writes the compact length: the entries of i_verify[b] before
// its first -1.
#include "common.cuh"
#include "kernels.h"

namespace dustin {

namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;
constexpr int kRows = 128;   // selected rows per CTA

__global__ void __launch_bounds__(kThreads) compact_kernel(const __grid_constant__ CompactArgs A) {
  pdl_launch_dependents();
  pdl_wait();
  const int nrun = (A.k + kRows - 1) / kRows;
  const int g = blockIdx.x / nrun, run = blockIdx.x - g * nrun, b = blockIdx.y, l = blockIdx.z;
  const CompactLayerDev& Ly = A.layer[l];
  int L = A.seq_len[b];
  if (L < 0 || L > A.Lcap) {
    if (threadIdx.x == 0 && g == 0 && run == 0 && l == 0) flag_error(A.err, DUSTIN_DEV_SEQLEN);
    L = 0;
  }
  const int32_t* I = A.ivf + size_t(b) * A.k;
  const int j0 = run * kRows;
  const int nr = min(kRows, A.k - j0);   // rows of this CTA
  const int chunks = A.D / 8;            // 16-byte chunks per row
  const int total = nr * chunks * 2;     // K rows, then V rows
  for (int base = threadIdx.x; base < total; base += kThreads * kBatch) {
    uint4 v[kBatch];
    int dst_row[kBatch], which[kBatch], ch[kBatch];
    bool live[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int q = base + u * kThreads;
      live[u] = q < total;
      const int w = q / (nr * chunks);
      const int rem = q - w * (nr * chunks);
      const int j = j0 + rem / chunks, c = rem - (rem / chunks) * chunks;
      which[u] = w;
      dst_row[u] = j;
      ch[u] = c;
      v[u] = make_uint4(0, 0, 0, 0);
      if (live[u]) {
        const int id = I[j];
        if (id >= 0 && id < L) {
          const uint16_t* src = w ? Ly.v + size_t(b) * Ly.vsb + size_t(g) * Ly.vsh + size_t(id) * Ly.vsl
                                  : Ly.k + size_t(b) * Ly.ksb + size_t(g) * Ly.ksh + size_t(id) * Ly.ksl;
          v[u] = __ldcs(reinterpret_cast<const uint4*>(src) + c);
        } else if (id != -1) {
          flag_error(A.err, DUSTIN_DEV_INDEX);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (!live[u]) continue;
      uint16_t* dst = which[u] ? Ly.vc + size_t(b) * Ly.vcsb + size_t(g) * Ly.vcsh + size_t(dst_row[u]) * Ly.vcsl
                               : Ly.kc + size_t(b) * Ly.kcsb + size_t(g) * Ly.kcsh + size_t(dst_row[u]) * Ly.kcsl;
      reinterpret_cast<uint4*>(dst)[ch[u]] = v[u];
    }
  }
  if (g == 0 && run == 0 && l == 0 && threadIdx.x < 32) {
    // the compact length: the entries before the first -1
    int first = A.k;
    for (int j0 = 0; j0 < A.k; j0 += 32) {
      const int j = j0 + int(threadIdx.x);
      const unsigned pad = __ballot_sync(0xffffffffu, j < A.k && I[j] == -1);
      if (pad) {
        first = j0 + __ffs(pad) - 1;
        break;
      }
    }
    if (threadIdx.x == 0) A.seq_len_c[b] = first;
  }
}

}  // namespace

cudaError_t compact_launch(const CompactArgs& a, cudaStream_t stream) {
  const int nrun = (a.k + kRows - 1) / kRows;
  return launch_pdl(compact_kernel, dim3(a.hkv * nrun, a.B, a.n_layers), dim3(kThreads), 0, stream, a);
}

}  // namespace dustin
