// Sparse and dense verification attention ("Technical Summary: Dustin",
// section 3 "Verification Workflow", steps 3-4; the dense comparator follows
// the "Problem Statement": standard verification loads the whole cache).
//
// Flash-decoding split-k on one GPU.  A cluster of CS CTAs covers one
// (layer, sequence b, KV head g); CTA s streams its share of the selected rows
// (sparse: the entries of I_verify; dense: positions 0..seq_len-1).  Rows are
// gathered with 1-D bulk copies (cp.async.bulk, one 2*D-byte row each) into
// padded shared-memory rows, so that ldmatrix reads are bank-conflict free.
// All (gamma+1) x G query rows that share the KV head are batched into
// 16-row m-tiles: S = Q K^T and O += P V run as bf16 m16n8k16 tensor-core
// MMAs with fp32 accumulation, one consumer warp per m-tile, with an online
// (log2-domain) softmax.  The last CTA of the cluster also attends to the
// gamma+1 draft-block rows under the causal mask u <= t.  The split partials
// (row max, row sum, unnormalised O) are merged by a log-sum-exp combine
// through distributed shared memory, so no partial ever goes to HBM.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace dustin {

namespace {

constexpr int TK = 64;  // keys per tile

template <int D>
struct VerifyGeom {
  static constexpr int RS = D * 2 + 16;   // padded row stride in bytes
  static constexpr int ROWB = D * 2;      // payload bytes per row
  static constexpr int OS = D + 4;        // partial-O row stride (floats)
};

template <int D, int MT, int NST>
struct VerifySmem {
  using Gm = VerifyGeom<D>;
  static constexpr size_t q_bytes = size_t(MT) * 16 * Gm::RS;
  static constexpr size_t stage_bytes = size_t(2) * TK * Gm::RS;
  static constexpr size_t ring_off = q_bytes;
  static constexpr size_t ring_bytes = NST * stage_bytes;
  static constexpr size_t partO_bytes = size_t(MT) * 16 * Gm::OS * 4;
  static constexpr size_t ring_alloc = ring_bytes > partO_bytes ? ring_bytes : partO_bytes;
  static constexpr size_t misc_off = ring_off + ring_alloc;
  // vmask[NST] | full[NST] | empty[NST] | qbar | part_m[MT*16] | part_l[MT*16] | abort
  static constexpr size_t misc_bytes = NST * 8 * 3 + 8 + size_t(MT) * 16 * 4 * 2 + 16;
  static constexpr size_t total = misc_off + misc_bytes;
};

template <int D, int MT, int NST>
__global__ void __launch_bounds__(32 * (MT + 1))
    verify_kernel(const __grid_constant__ VerifyArgs A) {
  using Gm = VerifyGeom<D>;
  using Sm = VerifySmem<D, MT, NST>;
  constexpr int RS = Gm::RS;
  constexpr int ROWB = Gm::ROWB;
  constexpr int NKS = D / 16;   // k-steps over the head dim
  constexpr int NOT = D / 8;    // 8-column n-tiles of O

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* Qs = smem;
  unsigned char* ring = smem + Sm::ring_off;
  uint64_t* vmask = reinterpret_cast<uint64_t*>(smem + Sm::misc_off);
  uint64_t* full = vmask + NST;
  uint64_t* empty = full + NST;
  uint64_t* qbar = empty + NST;
  float* part_m = reinterpret_cast<float*>(qbar + 1);
  float* part_l = part_m + MT * 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(part_l + MT * 16);
  float* part_O = reinterpret_cast<float*>(ring);  // reused after the main loop

  cg::cluster_group cluster = cg::this_cluster();
  const int CS = static_cast<int>(cluster.num_blocks());
  const int split = static_cast<int>(cluster.block_rank());
  const int g = blockIdx.y;
  const int layer = blockIdx.z / A.B;
  const int b = blockIdx.z % A.B;
  const VerifyLayerDev& Ly = A.layer[layer];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = A.T, G = A.G, NQ = A.NQ;

  int L = A.seq_len[b];
  if (L < 0 || L > A.Lcap) {
    if (threadIdx.x == 0 && split == 0 && g == 0 && layer == 0) flag_error(A.err, DUSTIN_DEV_SEQLEN);
    L = 0;
  }
  const int nkeys = A.dense ? L : A.k;
  const int base = split * A.keys_per_split;
  const int cnt = max(0, min(A.keys_per_split, nkeys - base));
  const int n_ctx_tiles = (cnt + TK - 1) / TK;
  const bool has_block = (split == CS - 1);
  const int n_tiles = n_ctx_tiles + (has_block ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], MT);
    }
    mbar_init(qbar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == MT) {
    // ------------------------------------------------------------ producer
    // Verify queries of this KV head: row r = t*G + hl (head g*G + hl).
    for (int r = NQ + lane; r < MT * 16; r += 32) {
      uint4* dst = reinterpret_cast<uint4*>(Qs + size_t(r) * RS);
      for (int c = 0; c < ROWB / 16; ++c) dst[c] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(qbar, uint32_t(NQ) * ROWB);
    __syncwarp();
    for (int r = lane; r < NQ; r += 32) {
      const int t = r / G, hl = r % G;
      const uint16_t* src = Ly.q + ((size_t(b) * T + t) * A.hq + size_t(g) * G + hl) * D;
      bulk_g2s(Qs + size_t(r) * RS, src, ROWB, qbar);
    }
    const uint64_t pol = policy_evict_first();
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i % NST;
      if (i >= NST) {
        if (!mbar_wait(&empty[s], ((i / NST) - 1) & 1, A.err, abort_flag)) break;
      }
      unsigned char* Kt = ring + size_t(s) * Sm::stage_bytes;
      unsigned char* Vt = Kt + size_t(TK) * RS;
      const bool blk = (i == n_ctx_tiles);
      int idx[2];
      bool ok[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int jj = lane + 32 * e;
        if (!blk) {
          const int j = base + i * TK + jj;
          const bool inr = j < base + cnt;
          int id = -1;
          if (inr) id = A.dense ? j : A.ivf[size_t(b) * A.k + j];
          ok[e] = inr && id >= 0 && id < L;
          if (inr && !A.dense && (id < -1 || id >= L)) flag_error(A.err, DUSTIN_DEV_INDEX);
          idx[e] = id;
        } else {
          ok[e] = jj < T;
          idx[e] = jj;
        }
      }
      const uint32_t m0 = __ballot_sync(0xffffffffu, ok[0]);
      const uint32_t m1 = __ballot_sync(0xffffffffu, ok[1]);
      if (lane == 0) vmask[s] = uint64_t(m0) | (uint64_t(m1) << 32);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if (!ok[e]) {
          uint4* dst = reinterpret_cast<uint4*>(Vt + size_t(lane + 32 * e) * RS);
          for (int c = 0; c < ROWB / 16; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async();
      __syncwarp();
      const uint32_t nvalid = __popc(m0) + __popc(m1);
      if (lane == 0) mbar_arrive_expect_tx(&full[s], nvalid * 2u * ROWB);
      __syncwarp();
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if (!ok[e]) continue;
        const int row = lane + 32 * e;
        const uint16_t *ks, *vs;
        if (blk) {
          const size_t off = ((size_t(b) * A.hkv + g) * T + idx[e]) * D;
          ks = Ly.kb + off;
          vs = Ly.vb + off;
        } else {
          ks = Ly.k + size_t(b) * Ly.ksb + size_t(g) * Ly.ksh + size_t(idx[e]) * Ly.ksl;
          vs = Ly.v + size_t(b) * Ly.vsb + size_t(g) * Ly.vsh + size_t(idx[e]) * Ly.vsl;
        }
        bulk_g2s_hint(Kt + size_t(row) * RS, ks, ROWB, &full[s], pol);
        bulk_g2s_hint(Vt + size_t(row) * RS, vs, ROWB, &full[s], pol);
      }
    }
  }

  // Consumer state (also needed by the partial write below).
  float o[NOT][4];
  float mrow[2] = {-INFINITY, -INFINITY};
  float lrow[2] = {0.f, 0.f};
#pragma unroll
  for (int n = 0; n < NOT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  if (warp < MT) {
    // ------------------------------------------------------------ consumers
    const int r0 = 16 * warp + (lane >> 2);
    const int t0 = r0 / G, t1 = (r0 + 8) / G;
    uint32_t qa[NKS][4];
    const bool qok = mbar_wait(qbar, 0, A.err, abort_flag);
    if (qok) {
      const uint32_t qbase = smem_u32(Qs);
#pragma unroll
      for (int ks = 0; ks < NKS; ++ks) {
        const int row = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int col = 16 * ks + 8 * (lane >> 4);
        ldmatrix_x4(qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], qbase + row * RS + col * 2);
      }
    }
    for (int i = 0; qok && i < n_tiles; ++i) {
      const int s = i % NST;
      if (!mbar_wait(&full[s], (i / NST) & 1, A.err, abort_flag)) break;
      const uint32_t Kt = smem_u32(ring + size_t(s) * Sm::stage_bytes);
      const uint32_t Vt = Kt + TK * RS;
      const uint64_t vm = vmask[s];
      const bool blk = (i == n_ctx_tiles);

      float sacc[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int ks = 0; ks < NKS; ks += 2) {
          uint32_t b0, b1, b2, b3;
          const int row = 8 * j + (lane & 7);
          const int col = 16 * ks + 8 * (lane >> 3);
          ldmatrix_x4(b0, b1, b2, b3, Kt + row * RS + col * 2);
          mma_bf16_16816(sacc[j], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma_bf16_16816(sacc[j], qa[ks + 1][0], qa[ks + 1][1], qa[ks + 1][2], qa[ks + 1][3], b2,
                         b3);
        }
      }
      // scale to the log2 domain and mask invalid keys
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = 8 * j + 2 * (lane & 3) + (e & 1);
          bool valid;
          if (blk) valid = key < T && key <= ((e >> 1) ? t1 : t0);
          else valid = (vm >> key) & 1ull;
          sacc[j][e] = valid ? sacc[j][e] * A.scale_log2 : -INFINITY;
        }
      }
      // online softmax (two rows per thread: r0 and r0 + 8)
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fmaxf(sacc[j][2 * hi], sacc[j][2 * hi + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mnew = fmaxf(mrow[hi], mx);
        const float basev = (mnew == -INFINITY) ? 0.f : mnew;
        const float alpha = exp2f(mrow[hi] - basev);
        mrow[hi] = mnew;
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
          for (int e = 2 * hi; e < 2 * hi + 2; ++e) {
            const float p = bf16_round(exp2f(sacc[j][e] - basev));
            sacc[j][e] = p;
            ls += p;
          }
        }
        lrow[hi] = lrow[hi] * alpha + ls;
#pragma unroll
        for (int n = 0; n < NOT; ++n) {
          o[n][2 * hi] *= alpha;
          o[n][2 * hi + 1] *= alpha;
        }
      }
      // O += P V
#pragma unroll
      for (int kk = 0; kk < TK / 16; ++kk) {
        const uint32_t a0 = pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]);
        const uint32_t a1 = pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]);
        const uint32_t a2 = pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
        const uint32_t a3 = pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) {
          uint32_t b0, b1, b2, b3;
          const int row = 16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int col = 16 * jj + 8 * (lane >> 4);
          ldmatrix_x4_trans(b0, b1, b2, b3, Vt + row * RS + col * 2);
          mma_bf16_16816(o[2 * jj], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(o[2 * jj + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
      lrow[hi] += __shfl_xor_sync(0xffffffffu, lrow[hi], 1);
      lrow[hi] += __shfl_xor_sync(0xffffffffu, lrow[hi], 2);
    }
  }

  // All copies have landed (or the CTA gave up): the ring becomes part_O.
  __syncthreads();
  if (warp < MT) {
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
      const int row = 16 * warp + (lane >> 2) + 8 * hi;
      if ((lane & 3) == 0) {
        part_m[row] = mrow[hi];
        part_l[row] = lrow[hi];
      }
      float* dst = part_O + size_t(row) * Gm::OS + 2 * (lane & 3);
#pragma unroll
      for (int n = 0; n < NOT; ++n)
        *reinterpret_cast<float2*>(dst + 8 * n) = make_float2(o[n][2 * hi], o[n][2 * hi + 1]);
    }
  }
  cluster.sync();

  // --------------------------------------------------- log-sum-exp combine
  constexpr int NW = MT + 1;
  constexpr int VPL = D / 32;   // floats per lane
  for (int rr = warp; ; rr += NW) {
    const int row = split + CS * rr;
    if (row >= NQ) break;
    float M = -INFINITY;
    for (int s = 0; s < CS; ++s) M = fmaxf(M, *cluster.map_shared_rank(part_m + row, s));
    const float basev = (M == -INFINITY) ? 0.f : M;
    float lsum = 0.f;
    float acc[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v) acc[v] = 0.f;
    for (int s = 0; s < CS; ++s) {
      const float w = exp2f(*cluster.map_shared_rank(part_m + row, s) - basev);
      lsum += w * *cluster.map_shared_rank(part_l + row, s);
      const float* src = cluster.map_shared_rank(part_O + size_t(row) * Gm::OS, s) + VPL * lane;
      if constexpr (VPL == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] += w * x.x; acc[1] += w * x.y;
      }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const int t = row / G, hl = row % G;
    float* dst = Ly.o + ((size_t(b) * T + t) * A.hq + size_t(g) * G + hl) * D + VPL * lane;
    if constexpr (VPL == 4) {
      *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    } else {
      *reinterpret_cast<float2*>(dst) = make_float2(acc[0] * inv, acc[1] * inv);
    }
  }
  cluster.sync();
}

template <int D, int MT, int NST>
cudaError_t launch_t(const VerifyArgs& a, const VerifyLaunch& pl, cudaStream_t stream) {
  auto kern = verify_kernel<D, MT, NST>;
  const size_t smem = VerifySmem<D, MT, NST>::total;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  if (pl.CS > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.CS, a.hkv, a.B * a.n_layers);
  cfg.blockDim = dim3(32 * (MT + 1));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int D, int NST>
cudaError_t launch_mt(const VerifyArgs& a, const VerifyLaunch& pl, cudaStream_t stream) {
  switch (pl.MT) {
    case 1: return launch_t<D, 1, NST>(a, pl, stream);
    case 2: return launch_t<D, 2, NST>(a, pl, stream);
    case 3: return launch_t<D, 3, NST>(a, pl, stream);
    case 4: return launch_t<D, 4, NST>(a, pl, stream);
    case 5: return launch_t<D, 5, NST>(a, pl, stream);
    case 6: return launch_t<D, 6, NST>(a, pl, stream);
    case 7: return launch_t<D, 7, NST>(a, pl, stream);
    case 8: return launch_t<D, 8, NST>(a, pl, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
size_t smem_for(int MT, int NST) {
#define DUSTIN_SM(mt, ns) \
  if (MT == mt && NST == ns) return VerifySmem<D, mt, ns>::total;
  DUSTIN_SM(1, 4) DUSTIN_SM(2, 4) DUSTIN_SM(3, 4) DUSTIN_SM(4, 4)
  DUSTIN_SM(5, 4) DUSTIN_SM(6, 4) DUSTIN_SM(7, 4) DUSTIN_SM(8, 4)
#undef DUSTIN_SM
  return 0;
}

}  // namespace

VerifyLaunch verify_plan(int D, int NQ, int nkeys_cap, int B, int hkv, int n_layers, int dense) {
  VerifyLaunch pl;
  pl.D = D;
  pl.MT = (NQ + 15) / 16;
  pl.NST = 4;   // the whole split of a sparse CTA (<= 4 tiles) is in flight at once
  // Split the keys of each (layer, b, g) over a cluster so that the grid
  // covers the GPU: aim for at least ~2 CTAs per SM in total.
  const int units = B * hkv * n_layers;
  const int max_splits = (nkeys_cap + TK - 1) / TK;
  int cs = 1;
  while (cs < 8 && units * cs < 2 * 152 && cs * 2 <= max_splits) cs *= 2;
  if (dense) cs = max_splits >= 8 ? 8 : cs;
  pl.CS = cs < 1 ? 1 : cs;
  pl.smem = D == 128 ? smem_for<128>(pl.MT, pl.NST) : smem_for<64>(pl.MT, pl.NST);
  return pl;
}

cudaError_t verify_launch(const VerifyArgs& a, const VerifyLaunch& pl, cudaStream_t stream) {
  if (pl.NST != 4) return cudaErrorInvalidValue;
  if (pl.D == 128) return launch_mt<128, 4>(a, pl, stream);
  if (pl.D == 64) return launch_mt<64, 4>(a, pl, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dustin
