// Hybrid importance scoring on Semantic Retrieval Heads ("Technical Summary:
// Dustin", section 1 "Hybrid Attention Aggregation" and section 2 "Efficient
// Estimation via Semantic Retrieval Heads").
//
// A "slab" is one (channel, layer, KV head g): every (SRH head of group g,
// query row) pair of that channel reads the same K rows.  For each sequence b
// the importance of position i in channel c is
//     sum over the slabs of c, sum over their pairs p of
//         exp(l_p,i - M_p) / S_p,   l = q.k / sqrt(d) (kept in the log2 domain)
// where M_p, S_p are the max and the sum of exp over the whole context.
//
// Kernel A (stream): the tiles of all (slab, sequence) pairs of a group of
// sequences form one sequence that is split evenly over one CTA per SM.  Each
// CTA streams its K rows once with 2-D TMA boxes (64 columns x 128 rows,
// 128-byte swizzle; 32 KB per tile) through a 6-stage mbarrier ring, computes
// the logits of all pairs at once with bf16 m16n8k16 MMAs (positions x
// pairs), writes them to a scratch buffer that stays in L2, and keeps an online
// (max, sum of exp) per pair for each contiguous segment of its range.
//
// Kernel B (normalise): per sequence, merges the segment statistics into
// M_p, S_p, then reads the logits back from L2, applies exp2(l - M_p) / S_p,
// sums over pairs and over the slabs of each channel and writes importance.
// It then discards the scratch lines from L2 so that they are never written
// back to HBM.  No attention tensor is materialised and K is read once.
#include "common.cuh"
#include "kernels.h"

namespace dustin {

namespace {

constexpr int kBoxCols = 64;
constexpr int kBoxRows = 128;
constexpr int kBoxBytes = kBoxCols * kBoxRows * 2;   // 16 KB
constexpr int kTileBytes = 2 * kBoxBytes;            // 128 rows x 128 or 256 rows x 64
constexpr int kStages = 6;
constexpr int kConsumers = 8;                        // 8 warps x 16 rows = 128 rows
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kMaxKs = 8;                            // d / 16 for d = 128
constexpr int kNormThreads = 256;                    // and positions per normalise CTA

__device__ __forceinline__ uint32_t tile_addr(uint32_t st, int D, int r, int c) {
  // element (row r, column c) of a tile stored as two TMA boxes of
  // [128 rows][128 bytes] with the 128-byte swizzle (chunk ^= row % 8)
  const int box = (D == 128) ? (c >> 6) : (r >> 7);
  const int chunk = (c & 63) >> 3;
  return st + box * kBoxBytes + (r & 127) * 128 + ((chunk ^ (r & 7)) << 4) + ((c & 7) << 1);
}

// Work is split by cost: CTA c owns the tiles whose cost prefix lies in
// [floor(c * W / G), floor((c + 1) * W / G)), W the total cost.

// Cost before flattened tile t.
__device__ __forceinline__ long long cost_prefix(const ScoreArgs& A, long long t) {
  int s = 0;
  while (s + 1 < A.n_slab && A.slab_start[s + 1] <= t) ++s;
  return A.cost_start[s] + (t - A.slab_start[s]) * A.slab[s].cost;
}

// First tile whose cost prefix is >= P.
__device__ __forceinline__ long long tile_at_cost(const ScoreArgs& A, long long P) {
  if (P >= A.total_cost) return A.total;
  int s = 0;
  while (s + 1 < A.n_slab && A.cost_start[s + 1] <= P) ++s;
  const long long k = (P - A.cost_start[s] + A.slab[s].cost - 1) / A.slab[s].cost;
  return A.slab_start[s] + k;
}

// CTA that owns flattened tile t.
__device__ __forceinline__ int owner_of(const ScoreArgs& A, long long t, int G) {
  const long long P = cost_prefix(A, t);
  return int(((P + 1) * G + A.total_cost - 1) / A.total_cost) - 1;
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Merges two (reference, sum of 2^(x - reference)) statistics.
__device__ __forceinline__ void stat_merge(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  s = (m == -INFINITY ? 0.f : s * exp2f(m - M)) + (m2 == -INFINITY ? 0.f : s2 * exp2f(m2 - M));
  m = M;
}

// Slab, sequence and tile of flattened tile t of the group (one division:
// called once per CTA; the walk then advances incrementally).
__device__ __forceinline__ void decode_tile(const ScoreArgs& A, long long t, int& s, int& bl,
                                            int& tile) {
  s = 0;
  while (s + 1 < A.n_slab && A.slab_start[s + 1] <= t) ++s;
  const long long off = t - A.slab_start[s];
  bl = int(off / A.slab[s].tiles);
  tile = int(off - (long long)bl * A.slab[s].tiles);
}

template <int D, int NTU, int NT>
__device__ __forceinline__ void consume_segment(const uint32_t (&qb)[NT][kMaxKs][2], float (&rm)[NT][2],
                                                float (&rs)[NT][2], unsigned char* ring,
                                                uint64_t* full, uint64_t* empty, int i0, int n,
                                                int r0, int L, int npairs, float* lrow, int LSP,
                                                int* err, volatile int* abort_flag) {
  constexpr int ROWS = (D == 128) ? kBoxRows : 2 * kBoxRows;
  constexpr int NMT = (D == 128) ? 1 : 2;
  constexpr int NKS = D / 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float scale = kLog2e * rsqrtf(float(D));
  // the logits are read once more, by the normalise kernel: keep them in L2
  // (the K rows stream through it with evict-first)
  const uint64_t keep = policy_evict_last();
  for (int k = 0; k < n; ++k, r0 += ROWS) {
    const int i = i0 + k;
    const int st = i % kStages;
    const bool ok = mbar_wait(&full[st], (i / kStages) & 1, err, abort_flag);
    if (ok && r0 < L) {
      const uint32_t sb = smem_u32(ring + size_t(st) * kTileBytes);
      const bool full_tile = r0 + ROWS <= L;
#pragma unroll
      for (int mi = 0; mi < NMT; ++mi) {
        const int rb = 16 * warp + kBoxRows * mi;
        float c[NTU][4];
#pragma unroll
        for (int j = 0; j < NTU; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
        const int arow = rb + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4(a0, a1, a2, a3, tile_addr(sb, D, arow, 16 * ks + 8 * (lane >> 4)));
#pragma unroll
          for (int j = 0; j < NTU; ++j)
            mma_bf16_16816(c[j], a0, a1, a2, a3, qb[j][ks][0], qb[j][ks][1]);
        }
        if (mi == NMT - 1) {   // the tile's shared memory is no longer read
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);
        }
        const int pos_lo = r0 + rb + (lane >> 2);
#pragma unroll
        for (int j = 0; j < NTU; ++j) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pair = 8 * j + 2 * (lane & 3) + (e & 1);
            const int pos = pos_lo + ((e >> 1) << 3);
            if (pair < npairs && (full_tile || pos < L)) {
              const float v = c[j][e] * scale;
              st_global_hint(lrow + size_t(pair) * LSP + pos, v, keep);
              // online sum of 2^(v - m) with a lazily raised reference m: the
              // reference only moves when v passes it by more than 8, so the
              // common path is one ex2 and one add
              float& m = rm[j][e & 1];
              float& sm = rs[j][e & 1];
              if (v > m + 8.f) {
                sm *= fast_exp2(m - v);
                m = v;
              }
              sm += fast_exp2(v - m);
            }
          }
        }
      }
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) score_stream_kernel(const __grid_constant__ ScoreArgs A) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* ring = smem;
  float* red = reinterpret_cast<float*>(smem + size_t(kStages) * kTileBytes);   // [8][32][2]
  uint64_t* full = reinterpret_cast<uint64_t*>(red + kConsumers * 32 * 2);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  // the range of this CTA (the group's tiles split by cost)
  const long long t0 = tile_at_cost(A, (long long)blockIdx.x * A.total_cost / G);
  const long long t1 = tile_at_cost(A, (long long)(blockIdx.x + 1) * A.total_cost / G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&A.map[0]);
  }
  if (A.wait_at_end) {
    pdl_launch_dependents();
  } else {
    pdl_wait();
    pdl_launch_dependents();   // the next launch may start once this one may run
  }
  // clear this group's selection histograms (the normalise kernel that
  // follows fills them; the selection of the previous call has completed)
  if (A.hist) {
    int* h = A.hist + size_t(A.b0) * 2 * kSelectBins;
    const int n = A.nb * 2 * kSelectBins;
    for (int j = blockIdx.x * kThreads + threadIdx.x; j < n; j += G * kThreads) h[j] = 0;
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ----------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int i = 0;
      // tiles [tile, tile + n) of (slab s, sequence bl) into the ring
      auto issue = [&](int s, int bl, int tile, int n) -> bool {
        const ScoreSlab& S = A.slab[s];
        const int b = A.b0 + bl;
        int L = A.seq_len[b];
        if (L < 0 || L > A.Lcap) L = 0;
        const int D = S.D, rows = S.rows, g = S.g, row2d = S.row2d;
        const CUtensorMap* map = &A.map[S.cache];
        const int rbase = row2d ? (b * row2d + g) * A.Lcap : 0;
        int r0 = tile * rows;
        for (int k = 0; k < n; ++k, ++i, r0 += rows) {
          const int st = i % kStages;
          if (i >= kStages && !mbar_wait(&empty[st], ((i / kStages) - 1) & 1, A.err, abort_flag)) return false;
          if (r0 >= L) {
            mbar_arrive(&full[st]);   // nothing to load: an empty tile
            continue;
          }
          unsigned char* dst = ring + size_t(st) * kTileBytes;
          auto load = [&](unsigned char* d, int x, int r) {
            if (row2d) tma_load_2d(d, map, x, rbase + r, &full[st], pol);
            else tma_load_4d(d, map, x, r, g, b, &full[st], pol);
          };
          if (D == 128) {
            mbar_arrive_expect_tx(&full[st], 2 * kBoxBytes);
            load(dst, 0, r0);
            load(dst + kBoxBytes, 64, r0);
          } else {
            const bool two = r0 + kBoxRows < L;
            mbar_arrive_expect_tx(&full[st], two ? 2 * kBoxBytes : kBoxBytes);
            load(dst, 0, r0);
            if (two) load(dst + kBoxBytes, 0, r0 + kBoxRows);
          }
        }
        return true;
      };
      bool ok = true;
      if (t0 < t1) {
        int s, bl, tile;
        decode_tile(A, t0, s, bl, tile);
        for (long long t = t0; t < t1 && ok;) {
          const int n = int(min((long long)(A.slab[s].tiles - tile), t1 - t));
          ok = issue(s, bl, tile, n);
          t += n;
          tile = 0;
          if (++bl == A.nb) {
            bl = 0;
            ++s;
          }
        }
      }
    }
  } else {
    // -------------------------------------------------------------- consumers
    uint32_t qb[NT][kMaxKs][2];
    float rm[NT][2], rs[NT][2];
    int i = 0;
    // tiles [tile, tile + n) of (slab s, sequence bl); statistics to slot
    auto segment = [&](int s, int bl, int tile, int n, int slot_idx) {
      const ScoreSlab& S = A.slab[s];
      const int b = A.b0 + bl;
      const int D = S.D, npairs = S.npairs;
      int L = A.seq_len[b];
      if (L < 0 || L > A.Lcap) {
        if (lane == 0 && warp == 0 && tile == 0) flag_error(A.err, DUSTIN_DEV_SEQLEN);
        L = 0;
      }
      // Q^T fragments (d x pairs) of this slab and sequence; fresh statistics
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int p = 8 * j + (lane >> 2);
        const uint16_t* qrow = nullptr;
        if (p < npairs) {
          const int hi = p / S.nq, tq = p - (p / S.nq) * S.nq;
          qrow = S.q + ((size_t(b) * S.nq + tq) * S.hq + S.heads[hi]) * D;
        }
#pragma unroll
        for (int ks = 0; ks < kMaxKs; ++ks) {
          uint32_t v0 = 0, v1 = 0;
          if (qrow && ks < (D >> 4)) {
            v0 = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * (lane & 3));
            v1 = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * (lane & 3));
          }
          qb[j][ks][0] = v0;
          qb[j][ks][1] = v1;
        }
        rm[j][0] = rm[j][1] = -INFINITY;
        rs[j][0] = rs[j][1] = 0.f;
      }
      float* lrow = A.logits + S.logit_off + size_t(bl) * npairs * A.LSP;
      const int ntu = (npairs + 7) >> 3;
      const int r0 = tile * S.rows;
#define DUSTIN_SEG(DD, NN)                                                                     \
  consume_segment<DD, NN, NT>(qb, rm, rs, ring, full, empty, i, n, r0, L, npairs, lrow, A.LSP, \
                              A.err, abort_flag)
      if (D == 128) {
        if (ntu <= 1) DUSTIN_SEG(128, 1);
        else if (ntu == 2 || NT < 3) DUSTIN_SEG(128, (NT < 2 ? NT : 2));
        else if (ntu == 3 || NT < 4) DUSTIN_SEG(128, (NT < 3 ? NT : 3));
        else DUSTIN_SEG(128, NT);
      } else {
        if (ntu <= 1) DUSTIN_SEG(64, 1);
        else if (ntu == 2 || NT < 3) DUSTIN_SEG(64, (NT < 2 ? NT : 2));
        else if (ntu == 3 || NT < 4) DUSTIN_SEG(64, (NT < 3 ? NT : 3));
        else DUSTIN_SEG(64, NT);
      }
#undef DUSTIN_SEG
      i += n;
      // segment statistics: reduce over lanes and warps, write one slot
#pragma unroll
      for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float m = rm[j][e], sm = rs[j][e];
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float s2 = __shfl_xor_sync(0xffffffffu, sm, o);
            stat_merge(m, sm, m2, s2);
          }
          const int pair = 8 * j + 2 * lane + e;
          if (lane < 4) {
            red[(warp * 32 + pair) * 2] = m;
            red[(warp * 32 + pair) * 2 + 1] = sm;
          }
        }
      }
      named_bar(1, 32 * kConsumers);
      if (warp == 0 && lane < npairs) {
        float m = -INFINITY, sm = 0.f;
        for (int w = 0; w < kConsumers; ++w)
          stat_merge(m, sm, red[(w * 32 + lane) * 2], red[(w * 32 + lane) * 2 + 1]);
        float* slot = A.stats + ((size_t(s) * A.nb + bl) * A.max_seg + slot_idx) * size_t(A.np_max) * 2;
        slot[lane * 2] = m;
        slot[lane * 2 + 1] = sm;
      }
      named_bar(1, 32 * kConsumers);
    };
    if (t0 < t1) {
      int s, bl, tile;
      decode_tile(A, t0, s, bl, tile);
      for (long long t = t0; t < t1;) {
        const int n = int(min((long long)(A.slab[s].tiles - tile), t1 - t));
        const long long first = A.slab_start[s] + (long long)bl * A.slab[s].tiles;
        segment(s, bl, tile, n, int(blockIdx.x) - owner_of(A, first, G));
        t += n;
        tile = 0;
        if (++bl == A.nb) {
          bl = 0;
          ++s;
        }
      }
    }
  }
  if (A.wait_at_end) pdl_wait();   // complete only after the previous launch
}

constexpr int kNormRowsMax = 48;   // logits rows staged per batch

// Adds one to h[bin] for every lane with ok: one reduction per distinct bin
// of the warp.
__device__ __forceinline__ void hist_red(int* h, uint32_t bin, bool ok, int lane) {
  const uint32_t mask = __match_any_sync(0xffffffffu, ok ? bin : 0xFFFFFFFFu);
  if (ok && lane == __ffs(mask) - 1) atomicAdd(h + bin, __popc(mask));
}

// CTA of the stream kernel that owns the tile whose cost prefix is P.
__device__ __forceinline__ int owner_at_cost(long long P, long long total_cost, int G) {
  return int(((P + 1) * G + total_cost - 1) / total_cost) - 1;
}

// Slab (index into the table) holding logits row r.
__device__ __forceinline__ int slab_of_row(const SlabInfo* si, int ns, int r) {
  int j = 0;
  while (j + 1 < ns && si[j + 1].row0 <= r) ++j;
  return j;
}

// Normalise kernel: over one or two stream launches' groups (a.ng), cps CTAs
// per sequence, each owning the 256-position chunks x = r, r + cps, ... of its
// sequence.  A work item is (chunk, batch of up to kNormRowsMax logits rows).
// Warp kNormWarps (the producer) bulk-copies each item's rows (one copy per
// row, completion on the buffer's full barrier) into one of two
// shared-memory buffers as soon as the compute warps have released it (their
// empty barrier), so no compute warp issues copies or waits on a block
// barrier.  Compute thread t owns position t of a chunk.
constexpr int kNormWarps = kNormThreads / 32;              // compute warps
constexpr int kNormBlock = kNormThreads + 32;              // plus the producer warp

__global__ void __launch_bounds__(kNormBlock, 2) score_norm_kernel(const __grid_constant__ ScoreArgs A) {
  // (the slab table is the only static shared memory; ptxas rounds it up to
  // whole KB, and the dynamic array starts after it)
  extern __shared__ __align__(128) unsigned char nsm[];
  __shared__ SlabInfo si[DUSTIN_MAX_SRH];
  const int nr = A.n_rows, n0 = A.n_rows0, ns = A.n_slab;
  const int nbr = nr < kNormRowsMax ? nr : kNormRowsMax;           // rows per batch
  float* lg = reinterpret_cast<float*>(nsm);                       // [2][nbr][256]
  float* Mg = lg + size_t(2) * nbr * kNormThreads;                 // [nr]
  float* Ig = Mg + nr;                                              // [nr]
  uint64_t* full = reinterpret_cast<uint64_t*>(Ig + nr);           // [2]; 2 nr floats above
  uint64_t* empty = full + 2;                                       // [2]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gr = (A.n_groups > 1 && int(blockIdx.x) >= A.ng[0].nb * A.ng[0].cps) ? 1 : 0;
  const NormGroup& NG = A.ng[gr];
  const int cps = NG.cps;
  const int cta = int(blockIdx.x) - (gr ? A.ng[0].nb * A.ng[0].cps : 0);
  const int bl = cta / cps, r = cta - (cta / cps) * cps;
  const int b = NG.b0 + bl;
  float* const logits = NG.logits;
  const int nchunks = (A.LSP + kNormThreads - 1) / kNormThreads;
  const int nbat = (nr + kNormRowsMax - 1) / kNormRowsMax;
  const int my_chunks = r < nchunks ? (nchunks - r + cps - 1) / cps : 0;
  const int n_items = my_chunks * nbat;
  // the slab table: one parameter word per thread, all loads in flight at once
  constexpr int kInfoWords = int(sizeof(SlabInfo) / 4);
  for (int j = tid; j < ns * kInfoWords; j += kNormBlock)
    reinterpret_cast<int*>(si)[j] = reinterpret_cast<const int*>(A.info[gr])[j];
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&empty[0], kNormWarps);
    mbar_init(&empty[1], kNormWarps);
    fence_barrier_init();
  }
  pdl_launch_dependents();
  pdl_wait();
  __syncthreads();
  // Item it = (chunk r + (it / nbat) cps, batch it % nbat) in buffer it % 2.
  // Logits row `row` of the item starting at position `base`.
  auto row_src = [&](int row, int base) -> const float* {
    const int j = slab_of_row(si, ns, row);
    return logits + si[j].logit_off + (size_t(bl) * si[j].npairs + (row - si[j].row0)) * A.LSP + base;
  };
  if (warp == kNormWarps) {
    // ------------------------------------------------------------- producer
    auto issue = [&](int it) {
      const int x = r + (it / nbat) * cps, k = it - (it / nbat) * nbat;
      const int r0 = k * kNormRowsMax, n = min(kNormRowsMax, nr - r0);
      const int base = x * kNormThreads, npos = min(kNormThreads, A.LSP - base);
      const int bf = it & 1;
      if (lane == 0) mbar_arrive_expect_tx(&full[bf], uint32_t(n) * uint32_t(npos) * 4u);
      __syncwarp();
      for (int q = lane; q < n; q += 32)
        bulk_g2s(lg + (size_t(bf) * nbr + q) * kNormThreads, row_src(r0 + q, base), uint32_t(npos) * 4,
                 &full[bf]);
    };
    // item 0 at once; item 1 once the statistics loads below have been served
    // (so that they do not queue behind its rows); then each item as soon as
    // its buffer is released
    if (n_items > 0) issue(0);
    named_bar(2, kNormBlock);
    for (int it = 1; it < n_items; ++it) {
      if (it >= 2 && !__all_sync(0xffffffffu, mbar_wait(&empty[it & 1], uint32_t((it >> 1) - 1) & 1u,
                                                          A.err, nullptr)))
        break;
      issue(it);
    }
    return;
  }
  // ------------------------------------------------------------- compute
  int L = A.seq_len[b];
  if (L < 0 || L > A.Lcap) L = 0;
  // merged statistics, one row per thread: M and 1 / S over the segments
  // (the CTAs owning the first to the last tile of (slab, sequence bl))
  for (int row = tid; row < nr; row += kNormThreads) {
    const int j = slab_of_row(si, ns, row);
    const int p = row - si[j].row0, tiles = si[j].tiles;
    const long long P0 = si[j].cost_start + (long long)bl * tiles * si[j].cost;
    const int seg0 = owner_at_cost(P0, NG.total_cost, NG.grid);
    const int n_seg = owner_at_cost(P0 + (long long)(tiles - 1) * si[j].cost, NG.total_cost, NG.grid) - seg0 + 1;
    const float* slots = NG.stats + (size_t(si[j].slab) * NG.nb + bl) * A.max_seg * size_t(A.np_max) * 2;
    float m = -INFINITY, sm = 0.f;
    for (int g = 0; g < n_seg; g += 4) {
      float2 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (g + u < n_seg) v[u] = __ldcg(reinterpret_cast<const float2*>(slots + (size_t(g + u) * A.np_max + p) * 2));
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (g + u < n_seg) stat_merge(m, sm, v[u].x, v[u].y);
    }
    Mg[row] = m;
    Ig[row] = sm > 0.f ? 1.f / sm : 0.f;
  }
  named_bar(2, kNormBlock);   // Mg, Ig complete (and the producer may issue item 1)
  const int s_eff = min(A.sinks, L);
  const int w0 = max(L - A.window, s_eff);
  int* h = A.hist ? A.hist + size_t(b) * 2 * kSelectBins : nullptr;
  float acc0 = 0.f, acc1 = 0.f;
  for (int it = 0; it < n_items; ++it) {
    const int bf = it & 1;
    const int x = r + (it / nbat) * cps, k = it - (it / nbat) * nbat;
    const int r0 = k * kNormRowsMax, n = min(kNormRowsMax, nr - r0);
    const int base = x * kNormThreads, npos = min(kNormThreads, A.LSP - base);
    if (!__all_sync(0xffffffffu, mbar_wait(&full[bf], uint32_t(it >> 1) & 1u, A.err, nullptr))) break;
    // row tid has landed: drop its lines from L2 without write-back (the
    // logits are dead once staged)
    if (tid < n) {
      const float* src = row_src(r0 + tid, base);
      for (int ln = 0; ln < npos * 4 / 128; ++ln)
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(src + ln * 32) : "memory");
    }
    if (tid < npos) {
      const float* lb = lg + size_t(bf) * nbr * kNormThreads + tid;
#pragma unroll 4
      for (int j = 0; j < n; ++j) {
        const int row = r0 + j;
        const float v = fast_exp2(lb[size_t(j) * kNormThreads] - Mg[row]) * Ig[row];
        if (row < n0) acc0 += v;
        else acc1 += v;
      }
    }
    // this warp is done with the buffer
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[bf]);
    if (k == nbat - 1) {   // the chunk's last batch: write it
      const int pos = base + tid;
      const bool live = pos < L;
      if (pos < A.Lcap) {
        A.importance[(size_t(b) * 2 + 0) * A.Lcap + pos] = live ? acc0 : 0.f;
        A.importance[(size_t(b) * 2 + 1) * A.Lcap + pos] = live ? acc1 : 0.f;
      }
      if (h) {
        const bool in_u = pos >= s_eff && pos < w0;
        // (positions past seq_len hold stale logits: they are never keyed)
        hist_red(h, in_u ? select_bin(importance_key(acc0, A.err)) : 0u, in_u, lane);
        hist_red(h + kSelectBins, in_u ? select_bin(importance_key(acc1, A.err)) : 0u, in_u, lane);
      }
      acc0 = acc1 = 0.f;
    }
  }
}

template <int NT>
cudaError_t launch_stream(const ScoreArgs& a, const ScoreLaunch& pl, cudaStream_t stream) {
  auto kern = score_stream_kernel<NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(pl.smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(a.grid), dim3(kThreads), pl.smem, stream, a);
}

}  // namespace

size_t score_stream_smem() {
  return size_t(kStages) * kTileBytes + kConsumers * 32 * 2 * 4 + kStages * 16 + 16 + 1024;
}

size_t score_norm_smem(int n_rows) {
  const int nb = n_rows < kNormRowsMax ? n_rows : kNormRowsMax;
  return size_t(2) * nb * kNormThreads * 4 + size_t(2 * n_rows) * 4 + 4 * 8 + 16;
}

// Shared-memory limit and carveout of the normalise kernel, set once: the
// largest layout, and all of the SM's unified memory as shared memory so that
// as many CTAs are resident as their shared memory allows.
static cudaError_t score_norm_attrs() {
  static const cudaError_t e = [] {
    cudaError_t r = cudaFuncSetAttribute(score_norm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(score_norm_smem(DUSTIN_MAX_SRH * DUSTIN_MAX_PAIRS)));
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(score_norm_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               int(cudaSharedmemCarveoutMaxShared));
    return r;
  }();
  return e;
}

int score_norm_ctas_per_sm(int n_rows) {
  // as the occupancy calculator counts them: registers, static and dynamic
  // shared memory, the carveout (a grid sized from the dynamic shared memory
  // alone can ask for more CTAs than fit, and the rest then run as a second
  // wave); the last answer per calling thread is kept (device, rows)
  static thread_local int last_dev = -1, last_rows = -1, last_n = 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev == last_dev && n_rows == last_rows) return last_n;
  int n = 0;
  if (score_norm_attrs() != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, score_norm_kernel, kNormBlock, score_norm_smem(n_rows)) !=
          cudaSuccess)
    return 1;
  last_dev = dev;
  last_rows = n_rows;
  last_n = n > 0 ? n : 1;
  return last_n;
}

int score_rows_per_tile(int D) { return D == 128 ? kBoxRows : 2 * kBoxRows; }

int score_tile_cost(int D, int npairs) {
  // 32 KB of K per tile plus the logits it writes (rows x pairs); the weight of
  // the logits term is the one that gave the shortest full score stage on the
  // 16-sequence, 32 K-position workload (heavier weights gave the same time)
  return 1000 + score_rows_per_tile(D) * npairs;
}

cudaError_t score_stream_launch(const ScoreArgs& a, const ScoreLaunch& pl, cudaStream_t stream) {
  switch (pl.NT) {
    case 1: return launch_stream<1>(a, pl, stream);
    case 2: return launch_stream<2>(a, pl, stream);
    case 3: return launch_stream<3>(a, pl, stream);
    case 4: return launch_stream<4>(a, pl, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t score_norm_launch(const ScoreArgs& a, const ScoreLaunch& pl, cudaStream_t stream) {
  const cudaError_t attr = score_norm_attrs();
  if (attr != cudaSuccess) return attr;
  int ctas = 0;
  for (int g = 0; g < a.n_groups; ++g) ctas += a.ng[g].nb * a.ng[g].cps;
  return launch_pdl(score_norm_kernel, dim3(ctas), dim3(kNormBlock), pl.norm_smem, stream, a);
}

}  // namespace dustin
