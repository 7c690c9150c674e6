// Sparse and dense verification attention ("Technical Summary: Dustin",
// section 3 "Verification Workflow", steps 3-4; the dense comparator follows
// the "Problem Statement": standard verification loads the whole cache).
//
// Work: for every (layer, sequence b, KV head g) "unit", the (gamma+1) x G
// query rows that share KV head g attend to the unit's key rows (sparse: the
// entries of I_verify; dense: positions 0..seq_len-1) plus the gamma+1
// draft-block rows under the causal mask u <= t.
//
// Schedule (stream-K): each unit is cut into 32-key tiles followed by one
// block tile; all units' tiles form one sequence that is split evenly over a
// grid sized to the GPU's resident capacity, so every CTA moves the same
// number of bytes whatever B, Hkv and k are.  A CTA walks its range one unit
// segment at a time.
//
// Data path: every warp issues 16-byte cp.async gathers (zero-filled for
// padding / out-of-context rows) into a 3-stage ring of 32-key tiles in padded
// shared-memory rows (2*d + 16 bytes, so ldmatrix is bank-conflict free); the
// index list runs one stage ahead through shared memory.  The ring is small so
// that several CTAs share an SM: cp.async reaches HBM bandwidth only with many
// resident warps.  Two warps share each 16-row m-tile of queries and take one
// half of every key tile: S = Q K^T and
// O += P V are bf16 m16n8k16 tensor-core MMAs with fp32 accumulation, with an
// online softmax in the log2 domain.
//
// Combine: a segment that covers a whole unit writes O directly; otherwise it
// writes (row max, row sum, unnormalised O) to the workspace and the last CTA
// to finish a segment of that unit (an atomic counter, no waiting) merges the
// segments with a log-sum-exp combine and resets the counter.
#include "common.cuh"
#include "kernels.h"

namespace dustin {

namespace {

constexpr int TK = 32;  // keys per tile: small stages so that ~3 CTAs share an SM
constexpr int NSTAGE = 3;
constexpr int TKH = TK / 2;   // keys per warp (each m-tile has two warps)

__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int D, int MT, int NST>
struct Lay {
  static constexpr int RS = D * 2 + 16;          // padded row stride (bytes)
  static constexpr int CH = D / 8;               // 16-byte chunks per row
  static constexpr int OS = D + 4;               // merge-area row stride (floats)
  static constexpr size_t q_off = 0;
  static constexpr size_t q_bytes = size_t(MT) * 16 * RS;
  static constexpr size_t stage_bytes = size_t(2) * TK * RS;
  static constexpr size_t ring_off = q_off + q_bytes;
  static constexpr size_t ring_bytes = NST * stage_bytes;
  static constexpr size_t merge_bytes = size_t(MT) * 16 * OS * 4 + size_t(MT) * 16 * 8;
  static constexpr size_t ring_alloc = ring_bytes > merge_bytes ? ring_bytes : merge_bytes;
  static constexpr size_t idx_off = ring_off + ring_alloc;
  static constexpr size_t idx_bytes = size_t(NST + 1) * TK * 4;
  static constexpr size_t misc_off = idx_off + idx_bytes;
  static constexpr size_t total = misc_off + 16;
};

// CTA that owns flattened tile x, for start(c) = c * total / G.
__device__ __forceinline__ int cta_of(long long x, long long total, int G) {
  return int(((x + 1) * G + total - 1) / total) - 1;
}

// Up to 3 resident CTAs per SM (96 threads per m-tile pair of warps at <= 112
// registers): the gathers of one CTA overlap the MMAs of the others.
template <int D, int MT, int NST>
__global__ void __launch_bounds__(64 * MT, MT <= 3 ? 3 : 1) verify_kernel(const __grid_constant__ VerifyArgs A) {
  using Ly = Lay<D, MT, NST>;
  constexpr int NTH = 64 * MT;
  constexpr int RS = Ly::RS;
  constexpr int CH = Ly::CH;
  constexpr int NKS = D / 16;
  constexpr int NOT = D / 8;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* Qs = smem + Ly::q_off;
  unsigned char* ring = smem + Ly::ring_off;
  int* idxs = reinterpret_cast<int*>(smem + Ly::idx_off);
  volatile int* s_last = reinterpret_cast<volatile int*>(smem + Ly::misc_off);
  float* mO = reinterpret_cast<float*>(ring);               // merge area (after drain)
  float* mM = mO + size_t(MT) * 16 * Ly::OS;
  float* mL = mM + MT * 16;

  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int mt = warp >> 1, half = warp & 1;
  const int G = gridDim.x;
  const long long total = A.total;
  const long long t0 = (long long)blockIdx.x * total / G;
  const long long t1 = (long long)(blockIdx.x + 1) * total / G;
  const int T = A.T, NQ = A.NQ, GQ = A.G;
  const int tiles_u = A.tiles_u, ctx_tiles = A.ctx_tiles;
  const int units_per_layer = A.B * A.hkv;

  for (long long t = t0; t < t1;) {
    const int u = int(t / tiles_u);
    const int ta = int(t % tiles_u);
    const long long rem_t = t1 - t;
    const int tb = int(rem_t < (long long)(tiles_u - ta) ? ta + rem_t : tiles_u);
    t += tb - ta;
    const int n = tb - ta;
    const int layer = u / units_per_layer;
    const int b = (u % units_per_layer) / A.hkv;
    const int g = u % A.hkv;
    const VerifyLayerDev& Lr = A.layer[layer];
    int L = A.seq_len[b];
    if (L < 0 || L > A.Lcap) {
      if (tid == 0 && g == 0 && layer == 0 && ta == 0) flag_error(A.err, DUSTIN_DEV_SEQLEN);
      L = 0;
    }
    const uint16_t* kbase = Lr.k + size_t(b) * Lr.ksb + size_t(g) * Lr.ksh;
    const uint16_t* vbase = Lr.v + size_t(b) * Lr.vsb + size_t(g) * Lr.vsh;
    const size_t blk_off = (size_t(b) * A.hkv + g) * T * D;

    // Key index of row r of local tile i, in two halves so that the global
    // load of I_verify is consumed one iteration after it is issued.
    auto raw_key = [&](int i, int r) -> int {
      const int tt = ta + i;
      if (tt >= ctx_tiles) return r;                     // draft-block tile
      const int j = tt * TK + r;
      if (A.dense) return j;
      return j < A.k ? __ldg(A.ivf + size_t(b) * A.k + j) : -1;
    };
    auto checked_key = [&](int i, int raw) -> int {       // -1: masked row
      const int tt = ta + i;
      if (tt >= ctx_tiles) return raw < T ? raw : -1;
      if (A.dense) return raw < L ? raw : -1;
      if (raw < -1 || raw >= L) {
        flag_error(A.err, DUSTIN_DEV_INDEX);
        return -1;
      }
      return raw;
    };
    auto issue_tile = [&](int i) {
      const int s = i % NST;
      const int* slot = idxs + (i % (NST + 1)) * TK;
      const bool blk = (ta + i) >= ctx_tiles;
      unsigned char* st = ring + size_t(s) * Ly::stage_bytes;
      for (int q = tid; q < 2 * TK * CH; q += NTH) {
        const int which = q / (TK * CH);
        const int rem = q - which * (TK * CH);
        const int row = rem / CH, ch = rem - (rem / CH) * CH;
        const int id = slot[row];
        const bool ok = id >= 0;
        const uint16_t* src;
        if (blk) src = (which ? Lr.vb : Lr.kb) + blk_off + size_t(ok ? id : 0) * D + ch * 8;
        else if (which) src = vbase + size_t(ok ? id : 0) * Lr.vsl + ch * 8;
        else src = kbase + size_t(ok ? id : 0) * Lr.ksl + ch * 8;
        cp_async16(st + size_t(which) * TK * RS + size_t(row) * RS + ch * 16, src, ok ? 16u : 0u);
      }
    };

    // ------------------------------------------------------------- prologue
    for (int q = tid; q < MT * 16 * CH; q += NTH) {
      const int r = q / CH, ch = q - (q / CH) * CH;
      unsigned char* dst = Qs + size_t(r) * RS + ch * 16;
      if (r < NQ) {
        const int tq = r / GQ, hl = r - (r / GQ) * GQ;
        cp_async16(dst, Lr.q + ((size_t(b) * T + tq) * A.hq + size_t(g) * GQ + hl) * D + ch * 8, 16u);
      } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    for (int i = 0; i < NST && i < n; ++i)
      if (tid < TK) idxs[(i % (NST + 1)) * TK + tid] = checked_key(i, raw_key(i, tid));
    int pf = (tid < TK && NST < n) ? raw_key(NST, tid) : -1;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NST - 1; ++i) {
      if (i < n) issue_tile(i);
      cp_async_commit();
    }

    float o[NOT][4];
#pragma unroll
    for (int x = 0; x < NOT; ++x) o[x][0] = o[x][1] = o[x][2] = o[x][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY};
    float lrow[2] = {0.f, 0.f};
    // A fragments are re-read from shared memory two k-steps at a time
    const uint32_t qb = smem_u32(Qs) + (16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1)) * RS + 16 * (lane >> 4);
    const int r0 = 16 * mt + (lane >> 2);
    const int tr0 = r0 / GQ, tr1 = (r0 + 8) / GQ;

    // ------------------------------------------------------------ main loop
    for (int i = 0; i < n; ++i) {
      cp_async_wait<NST - 2>();
      __syncthreads();
      if (tid < TK && i + NST < n) {
        idxs[((i + NST) % (NST + 1)) * TK + tid] = checked_key(i + NST, pf);
        pf = (i + NST + 1 < n) ? raw_key(i + NST + 1, tid) : -1;
      }
      if (i + NST - 1 < n) issue_tile(i + NST - 1);
      cp_async_commit();

      const uint32_t Kt = smem_u32(ring + size_t(i % NST) * Ly::stage_bytes);
      const uint32_t Vt = Kt + TK * RS;
      const int* slot = idxs + (i % (NST + 1)) * TK;
      const bool blk = (ta + i) >= ctx_tiles;
      const int kb0 = TKH * half;   // first key of this warp's half
      constexpr int NJ = TKH / 8;   // 8-key n-tiles per warp

      float sacc[NJ][4];
#pragma unroll
      for (int j = 0; j < NJ; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < NKS; ks += 2) {
        uint32_t qa[2][4];
        ldmatrix_x4(qa[0][0], qa[0][1], qa[0][2], qa[0][3], qb + ks * 32);
        ldmatrix_x4(qa[1][0], qa[1][1], qa[1][2], qa[1][3], qb + ks * 32 + 32);
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          uint32_t b0, b1, b2, b3;
          const int row = kb0 + 8 * j + (lane & 7);
          const int col = 16 * ks + 8 * (lane >> 3);
          ldmatrix_x4(b0, b1, b2, b3, Kt + row * RS + col * 2);
          mma_bf16_16816(sacc[j], qa[0][0], qa[0][1], qa[0][2], qa[0][3], b0, b1);
          mma_bf16_16816(sacc[j], qa[1][0], qa[1][1], qa[1][2], qa[1][3], b2, b3);
        }
      }
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kb0 + 8 * j + 2 * (lane & 3) + (e & 1);
          bool valid = slot[key] >= 0;
          if (blk) valid = valid && key <= ((e >> 1) ? tr1 : tr0);
          sacc[j][e] = valid ? sacc[j][e] * A.scale_log2 : -INFINITY;
        }
      }
      // Online softmax with a lazily moved reference: mrow is the reference
      // the exponentials are taken against; it only moves (and O and the row
      // sum are rescaled) when a tile's max passes it by more than 2^8, so
      // every p = 2^(s - mrow) stays <= 256 and most tiles skip the rescale.
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < NJ; ++j) mx = fmaxf(mx, fmaxf(sacc[j][2 * hi], sacc[j][2 * hi + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        if (mx > mrow[hi] + 8.f) {          // also the first tile with a valid key
          const float alpha = fast_exp2(mrow[hi] - mx);   // 0 while mrow is -inf
          mrow[hi] = mx;
          lrow[hi] *= alpha;
#pragma unroll
          for (int x = 0; x < NOT; ++x) {
            o[x][2 * hi] *= alpha;
            o[x][2 * hi + 1] *= alpha;
          }
        }
        const float basev = (mrow[hi] == -INFINITY) ? 0.f : mrow[hi];
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
#pragma unroll
          for (int e = 2 * hi; e < 2 * hi + 2; ++e) {
            const float p = bf16_round(fast_exp2(sacc[j][e] - basev));
            sacc[j][e] = p;
            ls += p;
          }
        }
        lrow[hi] += ls;
      }
#pragma unroll
      for (int kk = 0; kk < NJ / 2; ++kk) {
        const uint32_t a0 = pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]);
        const uint32_t a1 = pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]);
        const uint32_t a2 = pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
        const uint32_t a3 = pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) {
          uint32_t b0, b1, b2, b3;
          const int row = kb0 + 16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int col = 16 * jj + 8 * (lane >> 4);
          ldmatrix_x4_trans(b0, b1, b2, b3, Vt + row * RS + col * 2);
          mma_bf16_16816(o[2 * jj], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(o[2 * jj + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
      lrow[hi] += __shfl_xor_sync(0xffffffffu, lrow[hi], 1);
      lrow[hi] += __shfl_xor_sync(0xffffffffu, lrow[hi], 2);
    }
    cp_async_wait<0>();
    __syncthreads();   // ring is free: it becomes the merge area

    // ------------------------------------------- merge the two key halves
    if (half == 1) {
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        const int row = r0 + 8 * hi;
        if ((lane & 3) == 0) {
          mM[row] = mrow[hi];
          mL[row] = lrow[hi];
        }
        float* dst = mO + size_t(row) * Ly::OS + 2 * (lane & 3);
#pragma unroll
        for (int x = 0; x < NOT; ++x)
          *reinterpret_cast<float2*>(dst + 8 * x) = make_float2(o[x][2 * hi], o[x][2 * hi + 1]);
      }
    }
    __syncthreads();

    const int seg_first = cta_of((long long)u * tiles_u, total, G);
    const int seg_last = cta_of((long long)u * tiles_u + tiles_u - 1, total, G);
    const int n_seg = seg_last - seg_first + 1;
    const int seg = blockIdx.x - seg_first;
    const size_t slot_floats = size_t(A.slot_floats);   // NQ*D + 2*NQ, rounded to 4
    float* part = A.partial + (size_t(u) * A.max_seg + seg) * slot_floats;

    if (half == 0) {
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        const int row = r0 + 8 * hi;
        const float m1 = mM[row], l1 = mL[row];
        const float M = fmaxf(mrow[hi], m1);
        const float bv = (M == -INFINITY) ? 0.f : M;
        const float a0 = exp2f(mrow[hi] - bv), a1 = exp2f(m1 - bv);
        const float l = lrow[hi] * a0 + l1 * a1;
        const float* src = mO + size_t(row) * Ly::OS + 2 * (lane & 3);
        if (row < NQ) {
          if (n_seg == 1) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int tq = row / GQ, hl = row - (row / GQ) * GQ;
            float* dst = Lr.o + ((size_t(b) * T + tq) * A.hq + size_t(g) * GQ + hl) * D + 2 * (lane & 3);
#pragma unroll
            for (int x = 0; x < NOT; ++x) {
              const float2 h1 = *reinterpret_cast<const float2*>(src + 8 * x);
              *reinterpret_cast<float2*>(dst + 8 * x) =
                  make_float2((o[x][2 * hi] * a0 + h1.x * a1) * inv, (o[x][2 * hi + 1] * a0 + h1.y * a1) * inv);
            }
          } else {
            float* dst = part + size_t(row) * D + 2 * (lane & 3);
#pragma unroll
            for (int x = 0; x < NOT; ++x) {
              const float2 h1 = *reinterpret_cast<const float2*>(src + 8 * x);
              *reinterpret_cast<float2*>(dst + 8 * x) =
                  make_float2(o[x][2 * hi] * a0 + h1.x * a1, o[x][2 * hi + 1] * a0 + h1.y * a1);
            }
            if ((lane & 3) == 0) {
              part[size_t(NQ) * D + row] = M;
              part[size_t(NQ) * D + NQ + row] = l;
            }
          }
        }
      }
    }
    if (n_seg > 1) {
      __threadfence();
      __syncthreads();
      if (tid == 0) *s_last = (atomicAdd(&A.counters[u], 1) == n_seg - 1) ? 1 : 0;
      __syncthreads();
      if (*s_last) {
        __threadfence();
        const float* base0 = A.partial + size_t(u) * A.max_seg * slot_floats;
        for (int q = tid; q < NQ * (D / 4); q += NTH) {
          const int row = q / (D / 4), c4 = q - row * (D / 4);
          float M = -INFINITY;
          for (int s = 0; s < n_seg; ++s)
            M = fmaxf(M, __ldcg(base0 + s * slot_floats + size_t(NQ) * D + row));
          const float bv = (M == -INFINITY) ? 0.f : M;
          float lsum = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int s = 0; s < n_seg; ++s) {
            const float* ps = base0 + s * slot_floats;
            const float w = exp2f(__ldcg(ps + size_t(NQ) * D + row) - bv);
            lsum += w * __ldcg(ps + size_t(NQ) * D + NQ + row);
            const float4 x = __ldcg(reinterpret_cast<const float4*>(ps + size_t(row) * D) + c4);
            acc.x += w * x.x; acc.y += w * x.y; acc.z += w * x.z; acc.w += w * x.w;
          }
          const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
          const int tq = row / GQ, hl = row - (row / GQ) * GQ;
          float4* dst = reinterpret_cast<float4*>(
              Lr.o + ((size_t(b) * T + tq) * A.hq + size_t(g) * GQ + hl) * D) + c4;
          *dst = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
        if (tid == 0) A.counters[u] = 0;
      }
    }
    __syncthreads();   // merge area / idx slots are reused by the next segment
  }
}

template <int D, int MT>
cudaError_t launch_t(const VerifyArgs& a, const VerifyLaunch& pl, cudaStream_t stream) {
  auto kern = verify_kernel<D, MT, NSTAGE>;
  const size_t smem = Lay<D, MT, NSTAGE>::total;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(pl.grid), dim3(64 * MT), smem, stream, a);
}

template <int D, int MT>
int occupancy_t() {
  int n = 0;
  auto kern = verify_kernel<D, MT, NSTAGE>;
  const size_t smem = Lay<D, MT, NSTAGE>::total;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 64 * MT, smem) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

template <int D>
int occupancy_mt(int MT) {
  static int cache[9] = {};
  if (MT < 1 || MT > 8) return 1;
  if (!cache[MT]) {
    switch (MT) {
      case 1: cache[MT] = occupancy_t<D, 1>(); break;
      case 2: cache[MT] = occupancy_t<D, 2>(); break;
      case 3: cache[MT] = occupancy_t<D, 3>(); break;
      case 4: cache[MT] = occupancy_t<D, 4>(); break;
      case 5: cache[MT] = occupancy_t<D, 5>(); break;
      case 6: cache[MT] = occupancy_t<D, 6>(); break;
      case 7: cache[MT] = occupancy_t<D, 7>(); break;
      default: cache[MT] = occupancy_t<D, 8>(); break;
    }
  }
  return cache[MT];
}

template <int D>
cudaError_t launch_mt(const VerifyArgs& a, const VerifyLaunch& pl, cudaStream_t stream) {
  switch (pl.MT) {
    case 1: return launch_t<D, 1>(a, pl, stream);
    case 2: return launch_t<D, 2>(a, pl, stream);
    case 3: return launch_t<D, 3>(a, pl, stream);
    case 4: return launch_t<D, 4>(a, pl, stream);
    case 5: return launch_t<D, 5>(a, pl, stream);
    case 6: return launch_t<D, 6>(a, pl, stream);
    case 7: return launch_t<D, 7>(a, pl, stream);
    case 8: return launch_t<D, 8>(a, pl, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

VerifyLaunch verify_plan(int D, int NQ, int nkeys_cap, int B, int hkv, int n_layers, int dense,
                         int num_sms) {
  (void)dense;
  VerifyLaunch pl{};
  pl.D = D;
  pl.MT = (NQ + 15) / 16;
  pl.NST = NSTAGE;
  pl.ctx_tiles = (nkeys_cap + TK - 1) / TK;
  pl.tiles_u = pl.ctx_tiles + 1;
  pl.units = (long long)B * hkv * n_layers;
  pl.total = pl.units * pl.tiles_u;
  // as many CTAs as can be resident (several per SM)
  int occ = 1;
  if (num_sms > 0) occ = (D == 128) ? occupancy_mt<128>(pl.MT) : occupancy_mt<64>(pl.MT);
  long long grid = num_sms > 0 ? (long long)num_sms * occ : kVerifyGridMax;
  if (grid > kVerifyGridMax) grid = kVerifyGridMax;
  if (grid > pl.total) grid = pl.total;
  pl.grid = int(grid);
  // Partial slots per unit, bounded for any grid <= kVerifyGridMax: a unit of
  // tiles_u tiles meets at most tiles_u / per + 2 CTAs of >= per tiles each.
  const long long per = pl.total / kVerifyGridMax;
  pl.max_seg = int(pl.tiles_u / (per > 0 ? per : 1)) + 2;
  pl.slot_floats = ((long long)NQ * D + 2LL * NQ + 3) / 4 * 4;   // 16-byte aligned slots
  pl.smem = 0;
  return pl;
}

size_t verify_scratch_bytes(const VerifyLaunch& pl) {
  return size_t(pl.units) * pl.max_seg * size_t(pl.slot_floats) * 4;
}

cudaError_t verify_launch(const VerifyArgs& a, const VerifyLaunch& pl, cudaStream_t stream) {
  if (pl.D == 128) return launch_mt<128>(a, pl, stream);
  if (pl.D == 64) return launch_mt<64>(a, pl, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dustin
