// Budgeted tiered selection of I_verify ("Technical Summary: Dustin", section
// 1 "Hybrid Attention Aggregation": protect a sink prefix and a local window of
// recent tokens, then fill the rest of the fixed budget with the top-m tokens
// by the draft signal, then the most relevant remaining tokens by the target
// signal).
//
// One thread-block cluster of CS CTAs per sequence (CS = 8, 4, 2 or 1: the
// largest size whose B clusters are all resident at once); CTA r owns a
// contiguous slice of the unprotected positions.  Importance values are
// non-negative fp32, so their bit patterns order like the values.  Each tier
// finds the exact threshold key T of its top-cnt (descending key, ties to the
// lower index):
//   level 1  4096-bin histograms of the top 12 bits (sign, exponent and 3
//            mantissa bits) of both channels are built while the keys are
//            staged in shared memory; per tier they are merged across the
//            cluster through distributed shared memory (each rank merges one
//            slice of the bins), which gives the bin b1 that holds the cnt-th
//            key.  The draft tier's winners are taken out of the target
//            histogram as they are written.
//   pass A   one pass over the CTA's keys gathers the keys of bin b1 with their
//            positions and counts, per warp chunk, the keys above bin b1.
//   exact T  every CTA pulls all ranks' bin-b1 keys and finds T and the number
//            of keys equal to T that are taken with two local 10-bit radix
//            passes -- no cluster barrier -- and, from the same lists, how many
//            keys above T and equal to T lower ranks and lower warp chunks hold.
//   write    one ordered pass writes every key above T and the lowest-index
//            keys equal to T at their offsets (the draft tier also marks them
//            in a per-slice bitmap that the target tier skips).
// If the threshold bin holds more keys than the candidate lists take (heavy
// ties), T is found with histograms merged across the cluster instead, over
// the candidate lists where they fit and over whole slices where they do not.
#include <cooperative_groups.h>

#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace dustin {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins1 = 4096;      // top 12 bits
constexpr int kBins2 = 1024;      // 10 bits
constexpr int kCandCap = 2048;    // (key, position) candidates per CTA
constexpr int kPullCap = 4096;    // candidate keys of all ranks pulled into one CTA
constexpr int kBatch = 8;         // independent key loads in flight per thread
constexpr size_t kSmemBudget = 220 * 1024;

// CS: CTAs per sequence (the cluster size); rank r merges level-1 bins
// [r * 4096 / CS, (r + 1) * 4096 / CS)
template <int CS>
struct SelShared {
  static constexpr int kSliceBins = kBins1 / CS;
  static constexpr int kScratch = kSliceBins > kBins2 ? kSliceBins : kBins2;
  int h1[2][kBins1];         // level-1 histograms of this CTA's keys, per channel
  int gsl[kSliceBins];       // merged level-1 counts of this rank's bin slice
  int scratch[kScratch];     // a merged slice copy / local radix histograms
  union {
    uint32_t pulled[kPullCap];   // every rank's threshold-bin keys, in rank order
    int hist2[2][kBins2];        // or: cluster-merged refinement histograms (heavy ties)
  };
  uint32_t ckey[kCandCap];   // this CTA's keys of the threshold bin ...
  int cpos[kCandCap];        // ... and their positions
  int wabove[kWarps];        // per warp chunk: keys above the threshold bin
  int wgt[kWarps], weq[kWarps], wsum[kWarps];
  int rgt[CS], req[CS];      // per rank: pulled keys above / equal to T
  int poff[CS + 1];          // offsets of the ranks' lists in pulled
  int gsl_total, ncand, n_above;
  int bin, need, slice, need1;
  int gt_before, eq_before, cnt_gt, cnt_eq;
  int overflow;
};

__device__ __forceinline__ uint32_t key_of(float v, int* err) {
  const uint32_t u = __float_as_uint(v);
  if (v != v) {
    flag_error(err, DUSTIN_DEV_NAN);
    return 0u;
  }
  if (u & 0x80000000u) {
    if (u != 0x80000000u) flag_error(err, DUSTIN_DEV_NAN);
    return 0u;
  }
  return u;
}

struct KeySrc {
  const uint32_t* cached;  // shared-memory copy of the slice (indexed from its start)
  const float* global;     // importance row of this channel (indexed by position)
  int base;                // first position of the slice
  int* err;
  __device__ __forceinline__ uint32_t operator()(int i) const {
    return cached ? cached[i - base] : key_of(global[i], err);
  }
};

struct Excl {
  const uint32_t* bits;    // bitmap of the slice (bit i - base), or nullptr
  int base;
  __device__ __forceinline__ bool operator()(int i) const {
    if (!bits) return false;
    const int o = i - base;
    return (bits[o >> 5] >> (o & 31)) & 1u;
  }
};

// The slice [s0, s1) cut into one contiguous, 32-aligned chunk per warp (the
// order in which positions are written).
struct Chunks {
  int a0, chunk;
  __device__ Chunks(int s0, int s1) {
    a0 = s0 & ~31;
    chunk = (((s1 - a0 + kWarps - 1) / kWarps) + 31) & ~31;
    if (chunk == 0) chunk = 32;
  }
  __device__ __forceinline__ int of(int i) const { return (i - a0) / chunk; }
};

// Calls f(i, key, valid) for every i in [u0, u1), block-strided, kBatch loads
// in flight before use; every lane of every warp makes the same calls.
template <typename F>
__device__ __forceinline__ void for_keys(const KeySrc& key, int u0, int u1, const Excl& ex, F f) {
  for (int base = u0; base < u1; base += kThreads * kBatch) {
    uint32_t kv[kBatch];
    bool ok[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * kThreads + int(threadIdx.x);
      ok[u] = i >= key.base && i < u1 && !ex(i);
      kv[u] = ok[u] ? key(i) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) f(base + u * kThreads + int(threadIdx.x), kv[u], ok[u]);
  }
}

// Over hist[0..nbins) in descending bin order: the bin holding the need-th
// key, and how many keys of that bin are needed (written to sh.bin, sh.need).
// Whole-block call; nbins is a multiple of kThreads.
template <typename Sh>
__device__ void find_bin(Sh& sh, const int* hist, int nbins, int need) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = nbins / kThreads;
  int local = 0;
  for (int k = 0; k < q; ++k) local += hist[nbins - 1 - (tid * q + k)];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < kWarps ? sh.wsum[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kWarps) sh.wsum[lane] = wi - w;   // exclusive prefix
  }
  __syncthreads();
  const int before = sh.wsum[warp] + incl - local;
  if (before < need && need <= before + local) {
    int acc = before;
    for (int k = 0; k < q; ++k) {
      const int bin = nbins - 1 - (tid * q + k);
      const int h = hist[bin];
      if (acc + h >= need) {
        sh.bin = bin;
        sh.need = need - acc;
        break;
      }
      acc += h;
    }
  }
  __syncthreads();
}

// Heavy ties: the threshold key T below bin b1 from 10-bit histograms merged
// across the cluster (over the candidate lists where every CTA's fits, over
// the whole slice where it does not), then the per-warp and per-rank counts
// of keys above / equal to T.  Whole-cluster call; returns T, sets need.
template <int CS>
__device__ uint32_t slow_threshold(cg::cluster_group& cluster, const KeySrc& key, int s0, int s1,
                                   const Excl& ex, const Chunks& ck, uint32_t b1, int& need,
                                   SelShared<CS>& sh, int& hbuf) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = int(cluster.block_rank());
  const int ncand = sh.ncand;
  const bool listed = ncand <= kCandCap;
  uint32_t prefix = b1 << 20;
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = 10 - 10 * pass;
    const uint32_t hi_mask = 0xFFFFFFFFu << (shift + 10);
    int* h = sh.hist2[hbuf];
    for (int b = tid; b < kBins2; b += kThreads) h[b] = 0;
    __syncthreads();
    if (listed) {
      for (int c = tid; c < ncand; c += kThreads) {
        const uint32_t kv = sh.ckey[c];
        if ((kv & hi_mask) == prefix) atomicAdd(&h[(kv >> shift) & 1023u], 1);
      }
    } else {
      for_keys(key, s0, s1, ex, [&](int, uint32_t kv, bool ok) {
        if (ok && (kv & hi_mask) == prefix) atomicAdd(&h[(kv >> shift) & 1023u], 1);
      });
    }
    cluster.sync();
    for (int j = tid; j < kBins2; j += kThreads) {
      int v[CS];
#pragma unroll
      for (int q = 0; q < CS; ++q) v[q] = *cluster.map_shared_rank(&h[j], q);
      int g = 0;
#pragma unroll
      for (int q = 0; q < CS; ++q) g += v[q];
      sh.scratch[j] = g;
    }
    __syncthreads();
    find_bin(sh, sh.scratch, kBins2, need);
    prefix |= uint32_t(sh.bin) << shift;
    need = sh.need;
    hbuf ^= 1;   // the other buffer next: remote readers of this one may still run
  }
  const uint32_t T = prefix;
  // per-warp counts of keys above / equal to T in this CTA's chunks
  int ngt = 0, neq = 0;
  const int w0 = ck.a0 + warp * ck.chunk, w1 = min(w0 + ck.chunk, s1);
  for (int gb = w0; gb < w1; gb += 32 * kBatch) {
    uint32_t kv[kBatch];
    bool cv[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = gb + 32 * u + lane;
      cv[u] = i >= s0 && i < w1 && !ex(i);
      kv[u] = cv[u] ? key(i) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      ngt += __popc(__ballot_sync(0xffffffffu, cv[u] && kv[u] > T));
      neq += __popc(__ballot_sync(0xffffffffu, cv[u] && kv[u] == T));
    }
  }
  if (lane == 0) {
    sh.wgt[warp] = ngt;
    sh.weq[warp] = neq;
  }
  __syncthreads();
  if (tid == 0) {
    int g = 0, e = 0;
    for (int w = 0; w < kWarps; ++w) {
      g += sh.wgt[w];
      e += sh.weq[w];
    }
    sh.cnt_gt = g;
    sh.cnt_eq = e;
  }
  cluster.sync();
  if (tid == 0) {
    int g = 0, e = 0;
    for (int q = 0; q < rank; ++q) {
      g += *cluster.map_shared_rank(&sh.cnt_gt, q);
      e += *cluster.map_shared_rank(&sh.cnt_eq, q);
    }
    sh.gt_before = g;
    sh.eq_before = e;
  }
  __syncthreads();
  return T;
}

// Top `cnt` of the cluster's candidates (this CTA: [s0, s1) of key, minus ex)
// by (key desc, index asc), given this CTA's level-1 histogram h of them;
// writes this CTA's selected positions to out at its offset, and for the draft
// tier sets their bits in setbits and takes their target keys (sub) out of the
// target histogram.  Whole-cluster call.
template <int CS>
__device__ void tier_select(cg::cluster_group& cluster, const KeySrc& key, int s0, int s1,
                            const Excl& ex, int cnt, int* h, int32_t* out, uint32_t* setbits,
                            const KeySrc* sub, SelShared<CS>& sh, int& hbuf) {
  constexpr int kSliceBins = SelShared<CS>::kSliceBins;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = int(cluster.block_rank());
  if (cnt <= 0) return;   // same for every CTA of the cluster
  const Chunks ck(s0, s1);

  // ---- level 1: merge this rank's bin slice of every rank's histogram
  cluster.sync();                                   // A: every histogram complete
  // (ncand is reset only now: until every rank has passed barrier A, another
  // rank may still be reading this rank's previous candidate list)
  if (tid < kWarps) sh.wabove[tid] = 0;
  if (tid == 0) sh.ncand = 0;
  {
    int part = 0;
    for (int j = tid; j < kSliceBins; j += kThreads) {
      const int bin = rank * kSliceBins + j;
      int v[CS];
#pragma unroll
      for (int q = 0; q < CS; ++q) v[q] = *cluster.map_shared_rank(&h[bin], q);
      int g = 0;
#pragma unroll
      for (int q = 0; q < CS; ++q) g += v[q];
      sh.gsl[j] = g;
      part += g;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) sh.wsum[warp] = part;
    __syncthreads();
    if (tid == 0) {
      int t = 0;
      for (int w = 0; w < kWarps; ++w) t += sh.wsum[w];
      sh.gsl_total = t;
    }
  }
  cluster.sync();                                   // B: every slice merged
  if (tid == 0) {   // which rank's bin slice holds the cnt-th key (slices in descending order)
    int acc = 0;
    sh.slice = 0;
    sh.need1 = cnt;
    for (int q = CS - 1; q >= 0; --q) {
      const int t = *cluster.map_shared_rank(&sh.gsl_total, q);
      if (acc + t >= cnt) {
        sh.slice = q;
        sh.need1 = cnt - acc;
        break;
      }
      acc += t;
    }
  }
  __syncthreads();
  const int rs = sh.slice;
  for (int j = tid; j < kSliceBins; j += kThreads) sh.scratch[j] = *cluster.map_shared_rank(&sh.gsl[j], rs);
  __syncthreads();
  find_bin(sh, sh.scratch, kSliceBins, sh.need1);
  const uint32_t b1 = uint32_t(rs * kSliceBins + sh.bin);
  int need = sh.need;

  // ---- pass A: keys of bin b1 (with positions); per chunk, keys above bin b1
  // (walked from the 32-aligned slice start: a warp row of 32 positions lies in
  // one chunk, so the above-bin count takes one ballot and one atomic per row)
  const Excl exA{ex.bits, ex.base};
  for_keys(key, ck.a0, s1, exA, [&](int i, uint32_t kv, bool ok0) {
    const bool ok = ok0 && i >= s0;
    const uint32_t bin = kv >> 20;
    const uint32_t above = __ballot_sync(0xffffffffu, ok && bin > b1);
    if (above && lane == 0) atomicAdd(&sh.wabove[ck.of(i)], __popc(above));
    const bool hit = ok && bin == b1;
    const uint32_t ball = __ballot_sync(0xffffffffu, hit);
    if (ball) {
      int slot0 = 0;
      if (lane == 0) slot0 = atomicAdd(&sh.ncand, __popc(ball));
      slot0 = __shfl_sync(0xffffffffu, slot0, 0);
      const int slot = slot0 + __popc(ball & ((1u << lane) - 1u));
      if (hit && slot < kCandCap) {
        sh.ckey[slot] = kv;
        sh.cpos[slot] = i;
      }
    }
  });
  __syncthreads();
  if (tid == 0) {
    int a = 0;
    for (int w = 0; w < kWarps; ++w) a += sh.wabove[w];
    sh.n_above = a;
  }
  cluster.sync();                                   // C: candidate lists published
  if (tid == 0) {
    int off = 0, over = 0;
    for (int q = 0; q < CS; ++q) {
      const int n = *cluster.map_shared_rank(&sh.ncand, q);
      sh.poff[q] = off;
      if (n > kCandCap) over = 1;
      off += n;
    }
    sh.poff[CS] = off;
    sh.overflow = over || off > kPullCap;
  }
  __syncthreads();

  uint32_t T;
  if (!sh.overflow) {
    // ---- exact threshold from every rank's bin-b1 keys, locally
    const int total = sh.poff[CS];
#pragma unroll
    for (int q = 0; q < CS; ++q) {
      const int o = sh.poff[q], n = sh.poff[q + 1] - o;
      const uint32_t* src = cluster.map_shared_rank(sh.ckey, q);
      for (int j = tid; j < n; j += kThreads) sh.pulled[o + j] = src[j];
    }
    uint32_t prefix = b1 << 20;
    for (int pass = 0; pass < 2; ++pass) {
      const int shift = 10 - 10 * pass;
      const uint32_t hi_mask = 0xFFFFFFFFu << (shift + 10);
      for (int b = tid; b < kBins2; b += kThreads) sh.scratch[b] = 0;
      __syncthreads();
      for (int j = tid; j < total; j += kThreads) {
        const uint32_t kv = sh.pulled[j];
        if ((kv & hi_mask) == prefix) atomicAdd(&sh.scratch[(kv >> shift) & 1023u], 1);
      }
      __syncthreads();
      find_bin(sh, sh.scratch, kBins2, need);
      prefix |= uint32_t(sh.bin) << shift;
      need = sh.need;
    }
    T = prefix;
    // per rank and per warp chunk: keys above / equal to T
    if (tid < CS) {
      sh.rgt[tid] = 0;
      sh.req[tid] = 0;
    }
    if (tid < kWarps) {
      sh.wgt[tid] = sh.wabove[tid];
      sh.weq[tid] = 0;
    }
    __syncthreads();
    for (int j = tid; j < total; j += kThreads) {
      const uint32_t kv = sh.pulled[j];
      if (kv >= T) {
        int q = 0;
        while (j >= sh.poff[q + 1]) ++q;
        atomicAdd(kv > T ? &sh.rgt[q] : &sh.req[q], 1);
      }
    }
    const int ncand = sh.ncand;
    for (int c = tid; c < ncand; c += kThreads) {
      const uint32_t kv = sh.ckey[c];
      if (kv >= T) atomicAdd(kv > T ? &sh.wgt[ck.of(sh.cpos[c])] : &sh.weq[ck.of(sh.cpos[c])], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int g = 0, e = 0;
      for (int q = 0; q < rank; ++q) {
        g += *cluster.map_shared_rank(&sh.n_above, q) + sh.rgt[q];
        e += sh.req[q];
      }
      sh.gt_before = g;
      sh.eq_before = e;
    }
    __syncthreads();
  } else {
    T = slow_threshold(cluster, key, s0, s1, ex, ck, b1, need, sh, hbuf);
  }

  // ---- ordered write: every key above T and the lowest-index keys equal to T
  int gt_before = sh.gt_before, eq_before = sh.eq_before;
  for (int w = 0; w < warp; ++w) {
    gt_before += sh.wgt[w];
    eq_before += sh.weq[w];
  }
  int pos = gt_before + min(eq_before, need);
  int eq_run = eq_before;
  const uint32_t lt = (1u << lane) - 1u;
  const int w0 = ck.a0 + warp * ck.chunk, w1 = min(w0 + ck.chunk, s1);
  for (int gb = w0; gb < w1; gb += 32 * kBatch) {
    uint32_t kv[kBatch];
    bool cv[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = gb + 32 * u + lane;
      cv[u] = i >= s0 && i < w1 && !ex(i);
      kv[u] = cv[u] ? key(i) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int g0 = gb + 32 * u;
      const int i = g0 + lane;
      const bool isgt = cv[u] && kv[u] > T;
      const bool iseq = cv[u] && kv[u] == T;
      const uint32_t eqb = __ballot_sync(0xffffffffu, iseq);
      const bool sel = isgt || (iseq && (eq_run + __popc(eqb & lt)) < need);
      const uint32_t selb = __ballot_sync(0xffffffffu, sel);
      if (sel) {
        out[pos + __popc(selb & lt)] = i;
        if (sub) atomicAdd(&sh.h1[1][(*sub)(i) >> 20], -1);
      }
      // slice-local bitmap word of positions g0 .. g0 + 31 (g0 - a0 is 32-aligned)
      if (setbits && lane == 0 && g0 < w1) setbits[(g0 - ck.a0) >> 5] |= selb;
      pos += __popc(selb);
      eq_run += __popc(eqb);
    }
  }
  __syncthreads();
}

template <int CS>
__global__ void __launch_bounds__(kThreads, 2) select_kernel(const __grid_constant__ SelectArgs A) {
  extern __shared__ __align__(16) unsigned char dsm[];
  SelShared<CS>& sh = *reinterpret_cast<SelShared<CS>*>(dsm);
  unsigned char* rest = dsm + ((sizeof(SelShared<CS>) + 15) & ~size_t(15));
  pdl_launch_dependents();
  pdl_wait();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = int(cluster.block_rank());
  const int b = blockIdx.x / CS;
  const int tid = threadIdx.x;
  int32_t* out = A.out + size_t(b) * A.k;
  const int L = A.seq_len[b];
  // the early cases below are decided per sequence, so every CTA of the
  // cluster leaves together, before any cluster barrier
  if (L < 0 || L > A.Lcap) {
    if (tid == 0 && rank == 0) flag_error(A.err, DUSTIN_DEV_SEQLEN);
    for (int j = rank * kThreads + tid; j < A.k; j += CS * kThreads) out[j] = -1;
    return;
  }
  if (A.k >= L) {
    for (int j = rank * kThreads + tid; j < A.k; j += CS * kThreads) out[j] = j < L ? j : -1;
    return;
  }
  const int s_eff = min(A.sinks, L);
  const int w0 = max(L - A.window, s_eff);
  const int nP = s_eff + (L - w0);
  const int m1 = min(A.m, A.k - nP);
  const int f = A.k - nP - m1;
  if (rank == 0)
    for (int j = tid; j < nP; j += kThreads) out[j] = j < s_eff ? j : w0 + (j - s_eff);

  // this CTA's slice of the unprotected positions [s_eff, w0)
  const int per = (((w0 - s_eff) + CS - 1) / CS + 31) & ~31;
  const int s0 = min(w0, s_eff + rank * per);
  const int s1 = min(w0, s0 + per);
  const int nwords = (per + 63) / 32;   // bits of positions from (s0 & ~31)
  uint32_t* keys0 = A.cache_keys ? reinterpret_cast<uint32_t*>(rest) : nullptr;
  uint32_t* keys1 = A.cache_keys ? keys0 + A.slice_cap : nullptr;
  uint32_t* bitmap =
      reinterpret_cast<uint32_t*>(rest + (A.cache_keys ? size_t(2) * A.slice_cap * 4 : 0));
  for (int w = tid; w < nwords; w += kThreads) bitmap[w] = 0u;
  for (int j = tid; j < 2 * kBins1; j += kThreads) (&sh.h1[0][0])[j] = 0;
  int hbuf = 0;
  __syncthreads();

  // stage both channels' keys (when they fit) and build their level-1 histograms
  const float* row0 = A.imp + (size_t(b) * 2 + 0) * A.Lcap;
  const float* row1 = A.imp + (size_t(b) * 2 + 1) * A.Lcap;
  for (int base = s0; base < s1; base += kThreads * kBatch) {
    float v0[kBatch], v1[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * kThreads + tid;
      v0[u] = i < s1 ? row0[i] : 0.f;
      v1[u] = i < s1 ? row1[i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * kThreads + tid;
      if (i < s1) {
        const uint32_t k0 = key_of(v0[u], A.err), k1 = key_of(v1[u], A.err);
        if (keys0) {
          keys0[i - s0] = k0;
          keys1[i - s0] = k1;
        }
        atomicAdd(&sh.h1[0][k0 >> 20], 1);
        atomicAdd(&sh.h1[1][k1 >> 20], 1);
      }
    }
  }
  __syncthreads();
  const KeySrc src0{keys0, row0, s0, A.err}, src1{keys1, row1, s0, A.err};
  tier_select(cluster, src0, s0, s1, Excl{nullptr, 0}, m1, &sh.h1[0][0], out + nP, bitmap, &src1,
              sh, hbuf);
  tier_select(cluster, src1, s0, s1, Excl{bitmap, s0 & ~31}, f, &sh.h1[1][0], out + nP + m1,
              nullptr, static_cast<const KeySrc*>(nullptr), sh, hbuf);
  cluster.sync();   // no CTA leaves while another may still read its shared memory
}

template <int CS>
size_t smem_bytes(int slice_cap, int cache_keys) {
  return ((sizeof(SelShared<CS>) + 15) & ~size_t(15)) + (cache_keys ? size_t(2) * slice_cap * 4 : 0) +
         size_t(slice_cap + 64) / 32 * 4;
}

int slice_cap_of(int Lcap, int cs) { return int(size_t((Lcap + cs - 1) / cs + 31) & ~size_t(31)); }

// Shared-memory bytes of one CTA for cluster size CS; sets cache_keys and slice_cap.
template <int CS>
size_t plan_smem(SelectArgs& a) {
  a.slice_cap = slice_cap_of(a.Lcap, CS);
  a.cache_keys = smem_bytes<CS>(a.slice_cap, 1) <= kSmemBudget ? 1 : 0;
  return smem_bytes<CS>(a.slice_cap, a.cache_keys);
}

template <int CS>
cudaError_t launch_cs(const SelectArgs& a0, cudaStream_t stream, bool query_only, int* max_clusters) {
  SelectArgs a = a0;
  const size_t smem = plan_smem<CS>(a);
  auto kern = select_kernel<CS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.B * CS);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = CS;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  if (query_only) {
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(max_clusters, kern, &cfg);
  }
  return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_any(int cs, const SelectArgs& a, cudaStream_t stream, bool query_only, int* n) {
  switch (cs) {
    case 1: return launch_cs<1>(a, stream, query_only, n);
    case 2: return launch_cs<2>(a, stream, query_only, n);
    case 4: return launch_cs<4>(a, stream, query_only, n);
    case 8: return launch_cs<8>(a, stream, query_only, n);
    default: return cudaErrorInvalidValue;
  }
}

// How many clusters of cs CTAs can run at once for this Lcap on the current
// device (cached per device, cluster size and Lcap).
int max_active_clusters(int cs, const SelectArgs& a) {
  struct Entry {
    int dev, cs, Lcap, n;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.dev == dev && e.cs == cs && e.Lcap == a.Lcap) return e.n;
  int n = 0;
  if (launch_any(cs, a, nullptr, true, &n) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache.push_back({dev, cs, a.Lcap, n});
  return n;
}

}  // namespace

int select_cluster_size(const SelectArgs& a) {
  // the largest cluster whose B clusters are all resident at once; one CTA
  // per sequence when even pairs do not fit
  for (int cs = 8; cs >= 2; cs /= 2)
    if (a.B <= max_active_clusters(cs, a)) return cs;
  return 1;
}

cudaError_t select_launch(const SelectArgs& a, cudaStream_t stream) {
  return launch_any(select_cluster_size(a), a, stream, false, nullptr);
}

}  // namespace dustin
