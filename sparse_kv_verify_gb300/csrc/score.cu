// Hybrid importance scoring on Semantic Retrieval Heads ("Technical Summary:
// Dustin", section 1 "Hybrid Attention Aggregation" and section 2 "Efficient
// Estimation via Semantic Retrieval Heads").
//
// Work unit: a "slab" = one (channel, layer, KV head g) of one sequence b,
// together with every (SRH head of group g, query row) pair that reads it.
// A thread-block cluster of C CTAs covers the slab; CTA r owns positions
// [r*P, (r+1)*P) and
//   phase 1  streams its K rows once with 4-D TMA tiles (64 rows x 64 columns,
//            128-byte swizzle) through a 4-stage mbarrier ring, computes
//            logits l = q.k * log2(e)/sqrt(d) for all pairs at once as bf16
//            m16n8k16 MMAs (positions x pairs), keeps them in shared memory
//            and tracks per-pair maxima;
//   exchange the CTAs swap per-pair maxima, then per-pair sums of
//            exp2(l - M), through distributed shared memory;
//   phase 2  writes sum_pairs exp2(l - M_pair) / S_pair for each position: the
//            softmax normalisation and the sum over heads and query rows are
//            fused, and no attention tensor is ever written.
// A deterministic reduce then sums the per-slab maps of each channel in slab
// order into importance[B][2][Lcap].
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace dustin {

namespace {

constexpr int kRows = 64;              // positions per tile
constexpr int kBox = 64;               // bf16 columns per TMA box (128 bytes)
constexpr int kBoxBytes = kRows * kBox * 2;
constexpr int kStages = 4;
constexpr int kStageBytes = 2 * kBoxBytes;   // room for d = 128
constexpr int kConsumers = 4;          // 4 warps x 16 rows = one 64-row tile
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kMaxKs = 8;              // d / 16 for d = 128

struct ScoreSmemLayout {
  size_t ring = 0;                      // 1024-aligned
  size_t logits = 0;
  size_t small = 0;
  size_t total = 0;
};

__host__ __device__ inline ScoreSmemLayout score_layout(int np_max, int LS, bool smem_logits) {
  ScoreSmemLayout s;
  s.ring = 0;
  s.logits = size_t(kStages) * kStageBytes;
  const size_t lg = smem_logits ? size_t(np_max) * LS * 4 : 0;
  s.small = s.logits + lg;
  // red[4][32] | stat_m[32] | stat_s[32] | Mg[32] | inv[32] | full[4] | empty[4] | abort
  // +1024: the ring is aligned to 1024 bytes (128-byte swizzle atom) at run time
  s.total = s.small + (kConsumers * 32 + 4 * 32) * 4 + kStages * 16 + 16 + 1024;
  return s;
}

__device__ __forceinline__ uint32_t swz128(uint32_t stage, int row, int col) {
  // element (row, col) of a tile stored as d/64 boxes of [64 rows][128 bytes]
  // with the TMA 128-byte swizzle (16-byte chunk index XOR row % 8)
  const int box = col >> 6;
  const int chunk = (col & 63) >> 3;
  return stage + box * kBoxBytes + row * 128 + ((chunk ^ (row & 7)) << 4) + ((col & 7) << 1);
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int NT, bool SMEM_LOGITS>
__global__ void __launch_bounds__(kThreads, 1) score_kernel(const __grid_constant__ ScoreArgs A) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const ScoreSmemLayout lay = score_layout(A.np_max, A.LS, SMEM_LOGITS);
  unsigned char* ring = smem + lay.ring;
  float* red = reinterpret_cast<float*>(smem + lay.small);
  float* stat_m = red + kConsumers * 32;
  float* stat_s = stat_m + 32;
  float* Mg = stat_s + 32;
  float* inv = Mg + 32;
  uint64_t* full = reinterpret_cast<uint64_t*>(inv + 32);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);

  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int r = static_cast<int>(cluster.block_rank());
  const int si = blockIdx.y;
  const int b = blockIdx.z;
  const ScoreSlab& S = A.slab[si];
  const int D = S.D;
  const int nks = D >> 4;
  const int npairs = S.npairs;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  float* lg = SMEM_LOGITS
                  ? reinterpret_cast<float*>(smem + lay.logits)
                  : A.spill + ((size_t(si) * A.B + b) * C + r) * size_t(A.np_max) * A.LS;

  int L = A.seq_len[b];
  if (L < 0 || L > A.Lcap) {
    if (threadIdx.x == 0 && r == 0 && si == 0) flag_error(A.err, DUSTIN_DEV_SEQLEN);
    L = 0;
  }
  const int p0 = r * A.P;
  const int p1 = min(p0 + A.P, L);
  const int npos = max(0, p1 - p0);
  const int n_tiles = (npos + kRows - 1) / kRows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const float scale = kLog2e * rsqrtf(float(D));

  if (warp == kConsumers) {
    // ----------------------------------------------------------- TMA producer
    if (lane == 0 && n_tiles > 0) {
      const CUtensorMap* map = &A.map[S.cache];
      prefetch_tensormap(map);
      const uint64_t pol = policy_evict_first();
      const uint32_t bytes = uint32_t(D / kBox) * kBoxBytes;
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % kStages;
        if (i >= kStages) {
          if (!mbar_wait(&empty[s], ((i / kStages) - 1) & 1, A.err, abort_flag)) break;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        unsigned char* st = ring + size_t(s) * kStageBytes;
        for (int h = 0; h < D / kBox; ++h)
          tma_load_4d(st + h * kBoxBytes, map, h * kBox, p0 + i * kRows, S.g, b, &full[s], pol);
      }
    }
  } else {
    // -------------------------------------------------------------- consumers
    // B fragments of Q^T (d x pairs), loaded once: pair n = 8j + lane/4.
    uint32_t qb[NT][kMaxKs][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int p = 8 * j + (lane >> 2);
      const uint16_t* qrow = nullptr;
      if (p < npairs) {
        const int hi = p / S.nq, t = p % S.nq;
        qrow = S.q + ((size_t(b) * S.nq + t) * S.hq + S.heads[hi]) * D;
      }
#pragma unroll
      for (int ks = 0; ks < kMaxKs; ++ks) {
        uint32_t v0 = 0, v1 = 0;
        if (qrow && ks < nks) {
          v0 = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * (lane & 3));
          v1 = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * (lane & 3));
        }
        qb[j][ks][0] = v0;
        qb[j][ks][1] = v1;
      }
    }
    float runmax[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) runmax[j][0] = runmax[j][1] = -INFINITY;

    for (int i = 0; i < n_tiles; ++i) {
      const int s = i % kStages;
      if (!mbar_wait(&full[s], (i / kStages) & 1, A.err, abort_flag)) break;
      const uint32_t st = smem_u32(ring + size_t(s) * kStageBytes);
      float c[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
      const int arow = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int ks = 0; ks < kMaxKs; ++ks) {
        if (ks < nks) {
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4(a0, a1, a2, a3, swz128(st, arow, 16 * ks + 8 * (lane >> 4)));
#pragma unroll
          for (int j = 0; j < NT; ++j) mma_bf16_16816(c[j], a0, a1, a2, a3, qb[j][ks][0], qb[j][ks][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      // logits of positions lo = row lane/4 and hi = row lane/4 + 8 of this warp
      const int loc_lo = i * kRows + 16 * warp + (lane >> 2);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pair = 8 * j + 2 * (lane & 3) + (e & 1);
          const int loc = loc_lo + ((e >> 1) << 3);
          const float v = (loc < npos) ? c[j][e] * scale : -INFINITY;
          if (pair < npairs) {
            lg[size_t(pair) * A.LS + loc] = v;
            runmax[j][e & 1] = fmaxf(runmax[j][e & 1], v);
          }
        }
      }
    }
    // per-pair CTA maxima: lanes sharing lane%4 hold the same pairs
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = runmax[j][e];
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
        const int pair = 8 * j + 2 * lane + e;
        if (lane < 4 && pair < 32) red[warp * 32 + pair] = v;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int p = threadIdx.x;
    float v = -INFINITY;
    if (p < npairs)
      for (int w = 0; w < kConsumers; ++w) v = fmaxf(v, red[w * 32 + p]);
    stat_m[p] = v;
  }
  cluster.sync();  // exchange 1: maxima
  if (threadIdx.x < 32) {
    const int p = threadIdx.x;
    float M = -INFINITY;
    if (p < npairs)
      for (int q = 0; q < C; ++q) M = fmaxf(M, *cluster.map_shared_rank(stat_m + p, q));
    Mg[p] = M;
  }
  __syncthreads();
  // exponentiate in place and sum per pair (warp w takes pairs w, w+5, ...)
  for (int p = warp; p < npairs; p += kConsumers + 1) {
    const float M = Mg[p];
    float* row = lg + size_t(p) * A.LS;
    float acc = 0.f;
    for (int loc = lane; loc < npos; loc += 32) {
      const float e = (M == -INFINITY) ? 0.f : exp2f(row[loc] - M);
      row[loc] = e;
      acc += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) stat_s[p] = acc;
  }
  __syncthreads();
  cluster.sync();  // exchange 2: sums
  if (threadIdx.x < 32) {
    const int p = threadIdx.x;
    float Ssum = 0.f;
    if (p < npairs)
      for (int q = 0; q < C; ++q) Ssum += *cluster.map_shared_rank(stat_s + p, q);
    inv[p] = Ssum > 0.f ? 1.f / Ssum : 0.f;
  }
  cluster_arrive();  // remote reads of this CTA are done once everyone arrives
  __syncthreads();
  float* part = A.part + (size_t(si) * A.B + b) * A.Lcap + p0;
  for (int loc = threadIdx.x; loc < npos; loc += kThreads) {
    float acc = 0.f;
    for (int p = 0; p < npairs; ++p) acc += lg[size_t(p) * A.LS + loc] * inv[p];
    part[loc] = acc;
  }
  cluster_wait();
}

template <int NT, bool SM>
cudaError_t launch_t(const ScoreArgs& a, const ScoreLaunch& pl, cudaStream_t stream) {
  auto kern = score_kernel<NT, SM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(pl.smem));
  if (e != cudaSuccess) return e;
  if (pl.C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.C, a.n_slab, a.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <bool SM>
cudaError_t launch_nt(const ScoreArgs& a, const ScoreLaunch& pl, cudaStream_t stream) {
  switch (pl.NT) {
    case 1: return launch_t<1, SM>(a, pl, stream);
    case 2: return launch_t<2, SM>(a, pl, stream);
    case 3: return launch_t<3, SM>(a, pl, stream);
    case 4: return launch_t<4, SM>(a, pl, stream);
    default: return cudaErrorInvalidValue;
  }
}

__global__ void score_reduce_kernel(const __grid_constant__ ReduceArgs R) {
  const int c = blockIdx.y;
  const int b = blockIdx.z;
  const int pos = blockIdx.x * blockDim.x + threadIdx.x;
  if (pos >= R.Lcap) return;
  int L = R.seq_len[b];
  if (L < 0 || L > R.Lcap) L = 0;
  float v = 0.f;
  if (pos < L) {
    for (int s = 0; s < R.n_slab; ++s)
      if (R.channel_of[s] == c) v += R.part[(size_t(s) * R.B + b) * R.Lcap + pos];
  }
  R.importance[(size_t(b) * 2 + c) * R.Lcap + pos] = v;
}

}  // namespace

ScoreLaunch score_plan(int Lcap, int B, int n_slab, int np_max, int d_max) {
  (void)B;
  (void)n_slab;
  (void)d_max;
  ScoreLaunch pl{};
  pl.np_max = np_max;
  pl.NT = (np_max + 7) / 8;
  const size_t budget = 220 * 1024;
  for (int C : {8, 16}) {
    const int per = (Lcap + C - 1) / C;
    const int P = ((per + kRows - 1) / kRows) * kRows;
    const int LS = P + 4;
    const ScoreSmemLayout l = score_layout(np_max, LS, true);
    pl.C = C;
    pl.P = P;
    pl.LS = LS;
    if (l.total <= budget) {
      pl.smem_logits = true;
      pl.smem = l.total;
      pl.spill_bytes = 0;
      return pl;
    }
  }
  // logits too large for shared memory: keep them in a global scratch slice
  pl.smem_logits = false;
  pl.smem = score_layout(np_max, pl.LS, false).total;
  pl.spill_bytes = 0;  // caller multiplies per slab/sequence/CTA
  return pl;
}

cudaError_t score_launch(const ScoreArgs& a, const ScoreLaunch& pl, cudaStream_t stream) {
  return pl.smem_logits ? launch_nt<true>(a, pl, stream) : launch_nt<false>(a, pl, stream);
}

cudaError_t score_reduce_launch(const ReduceArgs& a, cudaStream_t stream) {
  dim3 grid((a.Lcap + 255) / 256, 2, a.B);
  score_reduce_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dustin
