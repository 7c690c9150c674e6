// Budgeted tiered selection of I_verify ("Technical Summary: Dustin", section
// 1 "Hybrid Attention Aggregation": protect a sink prefix and a local window of
// recent tokens, then fill the rest of the fixed budget with the top-m tokens
// by the draft signal, then the most relevant remaining tokens by the target
// signal).
//
// Importance values are non-negative fp32, so their bit patterns order like the
// values.  A tier takes the top cnt keys of its channel (descending key, ties
// to the lower position) among the unprotected positions U = [sinks, L -
// window) not taken by an earlier tier; the draft tier takes m1 keys of
// channel 0, the target tier f keys of channel 1.
//
// Input: 4096-bin histograms of the top 12 key bits of both channels over U,
// per sequence (built by the scoring kernel while it writes the importance,
// or by select_hist_kernel for a standalone call).
//
// select_kernel: one thread-block cluster of CS CTAs (1024 threads each) per
// sequence, each CTA owning one contiguous run of U (each warp a run of whole
// 128-position rows).
//   scan     every CTA finds, from the histograms, the bin b0 holding the m1-th
//            draft key and the bin b1 holding the (m1 + f)-th target key, and
//            in one pass (float4 loads) lists, in position order, the draft
//            keys of bins >= b0 (with the target key of the same position) and
//            the target keys of bins >= b1 of its run.  Every draft winner is
//            listed, and so is every target winner: the f-th target key
//            outside the draft tier is at least the (m1+f)-th target key of U,
//            because at most m1 of the top m1+f are taken by the draft tier.
//   finish   after a cluster barrier, rank 0 gathers every rank's lists through
//            distributed shared memory (a second barrier then lets the other
//            ranks leave) and selects exactly: draft tier -- two 10-bit radix
//            passes over the listed keys of bin b0 give the threshold key T and
//            how many keys equal to T are taken (the lowest positions), then
//            one ordered compaction of the list writes the tier; target tier
//            -- the same over the target list minus the draft tier, with the
//            target histogram corrected by the draft tier's target keys.
// When the level-1 histograms show that the lists of whole threshold bins
// would not fit rank 0's buffer (long sequences, large budgets), the list
// thresholds are first narrowed by the next 10 key bits: every CTA
// histograms those bits of its keys in the two threshold bins, rank 0 adds
// the CTAs' histograms through distributed shared memory and finds the
// sub-bins holding the m1-th draft and (m1 + f)-th target keys, and every CTA
// then lists only the keys at or above those sub-bins.  The finish is
// unchanged: it only needs every key at or above the tier's exact threshold.
// Every target entry also carries the draft key of its position, so once the
// draft tier's threshold key and tie cut are known, the target entries it
// took are marked by comparing keys.
// If a list outgrows its buffer (heavy ties), rank 0 selects that sequence
// with the general path:
// candidates of the threshold bin in a shared list (or, past its capacity,
// refinement over the whole range) and ordered passes over all keys.  Every
// path gives the same set.
#include <cooperative_groups.h>

#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace dustin {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins1 = kSelectBins;   // top 12 bits
constexpr int kBins2 = 1024;          // 10 bits per refinement pass
constexpr int kListCap = 128;         // entries per warp list and channel (scan)
constexpr int kCandCap = 4096;        // candidates of the general path
constexpr int kFinCap = 7424;         // list entries of both channels gathered by rank 0
constexpr int kBatch = 8;             // rows of 32 keys loaded before use (general path)
constexpr int kHistThreads = 1024;    // select_hist_kernel: positions per CTA
constexpr int kCells = kMaxSelectCtas * kWarps;   // (rank, warp) lists per channel

struct SelShared {
  int h[2][kBins1];          // level-1 histograms (h[0] holds the draft tier's
                             // positions once the scan is done)
  int h2[kBins2];            // refinement histogram
  union {
    struct {                 // scan: per-warp ordered lists
      uint32_t k0[kWarps][kListCap];    // draft keys ...
      uint32_t k0t[kWarps][kListCap];   // ... the target keys of their positions ...
      int p0[kWarps][kListCap];         // ... and the positions
      uint32_t k1[kWarps][kListCap];    // target keys ...
      int p1[kWarps][kListCap];         // ... positions ...
      uint32_t k1d[kWarps][kListCap];   // ... and the draft keys of those positions
    } l;
    struct {                 // general path: threshold-bin candidates
      uint32_t key[kCandCap];
      int pos[kCandCap];
    } c;
    int r2[2][kBins2];       // list refinement: next 10 bits of the threshold bins
  } u;
  // rank 0: the gathered lists, draft entries [0, n0) then target [n0, n0 + n1)
  uint32_t ekey[kFinCap];
  int epos[kFinCap];
  uint32_t ek0t[kFinCap];    // draft entry: its target key; target entry: its draft key
  int cell[2][kCells + 1];   // list counts, then offsets, per (rank, warp); then the total
  int ovf_all[kCells];       // per (rank, warp): its list overflowed
  int wsum[kWarps];          // scan scratch
  int wgt[kWarps], weq[kWarps];   // per warp: keys above / equal to T
  int gtb[kWarps], eqb[kWarps];   // exclusive prefixes of wgt, weq
  int ncand, bin, need, found, overflow;
  int wsum2[2][kWarps];      // find_bin2 scratch and results, per histogram
  int bin2[2], need2[2], found2[2];
  uint32_t t_draft;          // the draft tier's threshold key ...
  int tie_cut;               // ... and the last position taken at that key
  uint32_t thr[2];           // rank 0: refined list thresholds (keys) of both channels
};
static_assert(sizeof(SelShared) + 16 <= 227 * 1024, "select state must fit one CTA's shared memory");

// ------------------------------------------------------------------ helpers

// Split cluster barrier: a CTA arrives early and waits later; once the wait
// returns, every CTA of the cluster has started (its shared memory may be
// written by the others).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait;" ::: "memory"); }

// Key of position i of one channel's importance row.
struct Keys {
  const float* row;
  int* err;
  __device__ __forceinline__ uint32_t operator()(int i) const { return importance_key(__ldg(row + i), err); }
};

// Positions taken by the draft tier (general path): bit (i - b0) of a bitmap.
struct Excl {
  const uint32_t* bits;
  int b0;
  __device__ __forceinline__ bool operator()(int i) const {
    if (!bits) return false;
    const int o = i - b0;
    return (bits[o >> 5] >> (o & 31)) & 1u;
  }
};

// [s0, s1) cut into one contiguous run of whole 32-position rows per warp,
// starting at the 32-aligned a0 <= s0.
struct Chunks {
  int s0, s1, a0, chunk;
  __device__ Chunks(int s0_, int s1_) : s0(s0_), s1(s1_) {
    a0 = s0 & ~31;
    chunk = ((((s1 - a0) + kWarps - 1) / kWarps) + 31) & ~31;
    if (chunk <= 0) chunk = 32;
  }
  __device__ __forceinline__ int w0(int w) const { return a0 + w * chunk; }
  __device__ __forceinline__ int w1(int w) const { return min(a0 + (w + 1) * chunk, s1); }
  __device__ __forceinline__ int warp_of(int i) const { return (i - a0) / chunk; }
};

// Adds one to h[bin] for every lane with ok, one atomic per distinct bin of
// the warp (h in shared or global memory).
__device__ __forceinline__ void hist_add(int* h, uint32_t bin, bool ok, int lane) {
  const uint32_t mask = __match_any_sync(0xffffffffu, ok ? bin : 0xFFFFFFFFu);
  if (ok && lane == __ffs(mask) - 1) atomicAdd(&h[bin], __popc(mask));
}

// Calls f(i, key, ok) for every position of this warp's rows of 32 (general
// path); ok = i in [s0, s1) and not excluded.  kBatch rows in flight.
template <typename F>
__device__ __forceinline__ void for_rows(const Keys& key, const Chunks& ck, const Excl& ex, F f) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w0 = ck.w0(warp), w1 = ck.w1(warp);
  for (int gb = w0; gb < w1; gb += 32 * kBatch) {
    uint32_t kv[kBatch];
    bool ok[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = gb + 32 * u + lane;
      ok[u] = i >= ck.s0 && i < w1 && !ex(i);
      kv[u] = ok[u] ? key(i) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (gb + 32 * u < w1) f(gb + 32 * u + lane, kv[u], ok[u]);
  }
}

// Over hist[0..nbins) in descending bin order: the bin holding the need-th
// key and how many keys of it are needed (sh.bin, sh.need; sh.found = 0 if the
// histogram holds fewer than need keys).  Whole-block call.
__device__ void find_bin(SelShared& sh, const int* hist, int nbins, int need) {
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
  if (tid == 0) sh.found = 0;
  __syncthreads();
  if (warp == 0) {
    const int w = sh.wsum[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    sh.wsum[lane] = wi - w;   // exclusive prefix
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
        sh.found = 1;
        break;
      }
      acc += h;
    }
  }
  __syncthreads();
}

// find_bin over the two level-1 histograms at once (one set of block
// barriers): for c = 0, 1 with need_c > 0, the bin of h_c holding the
// need_c-th key and how many keys of it are needed (sh.bin2[c], sh.need2[c];
// sh.found2[c] = 0 if h_c holds fewer keys).  Whole-block call.
__device__ void find_bin2(SelShared& sh, const int* h0, int need0, const int* h1, int need1) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int q = kBins1 / kThreads;
  int loc[2] = {0, 0};
#pragma unroll
  for (int k = 0; k < q; ++k) {
    const int bin = kBins1 - 1 - (tid * q + k);
    loc[0] += h0[bin];
    loc[1] += h1[bin];
  }
  int incl[2] = {loc[0], loc[1]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int y = __shfl_up_sync(0xffffffffu, incl[c], o);
      if (lane >= o) incl[c] += y;
    }
  }
  if (lane == 31) {
    sh.wsum2[0][warp] = incl[0];
    sh.wsum2[1][warp] = incl[1];
  }
  if (tid < 2) sh.found2[tid] = 0;
  __syncthreads();
  if (warp < 2) {   // warp c: exclusive prefix of histogram c's warp sums
    const int w = sh.wsum2[warp][lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    sh.wsum2[warp][lane] = wi - w;
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int need = c ? need1 : need0;
    const int* h = c ? h1 : h0;
    const int before = sh.wsum2[c][warp] + incl[c] - loc[c];
    if (need > 0 && before < need && need <= before + loc[c]) {
      int acc = before;
      for (int k = 0; k < q; ++k) {
        const int bin = kBins1 - 1 - (tid * q + k);
        if (acc + h[bin] >= need) {
          sh.bin2[c] = bin;
          sh.need2[c] = need - acc;
          sh.found2[c] = 1;
          break;
        }
        acc += h[bin];
      }
    }
  }
  __syncthreads();
}

// Exclusive prefixes of the per-warp counts wgt, weq into gtb, eqb.
__device__ void warp_prefixes(SelShared& sh) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    const int g = sh.wgt[tid], e = sh.weq[tid];
    int gi = g, ei = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, gi, o);
      const int z = __shfl_up_sync(0xffffffffu, ei, o);
      if (tid >= o) {
        gi += y;
        ei += z;
      }
    }
    sh.gtb[tid] = gi - g;
    sh.eqb[tid] = ei - e;
  }
  __syncthreads();
}

// Two 10-bit radix passes below the 12-bit prefix b1: the exact threshold key
// T and, in *need, how many keys equal to T are taken.  visit(f) calls
// f(key, ok) for every candidate key (keys outside bin b1 must have ok false).
template <typename V>
__device__ uint32_t refine(SelShared& sh, uint32_t b1, int* need, V visit) {
  uint32_t prefix = b1 << 20;
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = 10 - 10 * pass;
    const uint32_t hi_mask = 0xFFFFFFFFu << (shift + 10);
    sh.h2[threadIdx.x] = 0;
    __syncthreads();
    visit([&](uint32_t kv, bool ok) {
      if (ok && (kv & hi_mask) == prefix) atomicAdd(&sh.h2[(kv >> shift) & 1023u], 1);
    });
    __syncthreads();
    find_bin(sh, sh.h2, kBins2, *need);
    prefix |= uint32_t(sh.bin) << shift;
    *need = sh.need;
  }
  return prefix;
}

// Writes one selected position: its slot (guarded: a histogram that disagreed
// with the keys could otherwise push it past the tier), the draft tier's
// bitmap bit and its target key taken out of the target histogram.
struct Emit {
  int32_t* out;
  int cnt;
  uint32_t* bits;    // draft tier: bitmap to mark, else nullptr
  int b0;
  const Keys* sub1;  // draft tier: target keys to take out, else nullptr
  int* h1;
  int* err;
  __device__ __forceinline__ void operator()(int o, int i) const {
    if (o < cnt) out[o] = i;
    else flag_error(err, DUSTIN_DEV_NAN);
    if (bits) atomicOr(&bits[(i - b0) >> 5], 1u << ((i - b0) & 31));
    if (sub1) atomicSub(&h1[select_bin((*sub1)(i))], 1);
  }
};

// ----------------------------------------------------------- general path

// One tier over the whole range [s0, s1) minus ex, given the level-1
// histogram h of exactly those keys.
__device__ void tier_general(SelShared& sh, const Keys& key, const Excl& ex, int s0, int s1, int cnt,
                             const int* h, const Emit& emit, int* err) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lt = (1u << lane) - 1u;
  const Chunks ck(s0, s1);
  find_bin(sh, h, kBins1, cnt);
  if (!sh.found) {   // inconsistent histogram: cannot happen with matching keys
    if (tid == 0) flag_error(err, DUSTIN_DEV_NAN);
    for (int j = tid; j < cnt; j += kThreads) emit.out[j] = -1;
    __syncthreads();
    return;
  }
  const uint32_t b1 = uint32_t(sh.bin);
  int need = sh.need;
  if (tid == 0) sh.ncand = 0;
  __syncthreads();

  // ---- pass A: keys above bin b1 per warp; the keys of bin b1
  int above = 0;
  for_rows(key, ck, ex, [&](int i, uint32_t kv, bool ok) {
    const uint32_t bin = select_bin(kv);
    above += __popc(__ballot_sync(0xffffffffu, ok && bin > b1));
    const bool hit = ok && bin == b1;
    const uint32_t ball = __ballot_sync(0xffffffffu, hit);
    if (ball) {
      int slot0 = 0;
      if (lane == 0) slot0 = atomicAdd(&sh.ncand, __popc(ball));
      slot0 = __shfl_sync(0xffffffffu, slot0, 0);
      const int slot = slot0 + __popc(ball & lt);
      if (hit && slot < kCandCap) {
        sh.u.c.key[slot] = kv;
        sh.u.c.pos[slot] = i;
      }
    }
  });
  if (lane == 0) {
    sh.wgt[warp] = above;
    sh.weq[warp] = 0;
  }
  __syncthreads();
  const int ncand = sh.ncand;
  const bool listed = ncand <= kCandCap;

  // ---- refine
  const uint32_t T = refine(sh, b1, &need, [&](auto f) {
    if (listed) {
      for (int c = tid; c < ncand; c += kThreads) f(sh.u.c.key[c], true);
    } else {
      for_rows(key, ck, ex, [&](int, uint32_t kv, bool ok) { f(kv, ok && select_bin(kv) == b1); });
    }
  });
  const int need_eq = need;

  // ---- per warp chunk: keys of bin b1 above / equal to T
  if (listed) {
    for (int c = tid; c < ncand; c += kThreads) {
      const uint32_t kv = sh.u.c.key[c];
      const int w = ck.warp_of(sh.u.c.pos[c]);
      if (kv >= T) atomicAdd(kv > T ? &sh.wgt[w] : &sh.weq[w], 1);
    }
  } else {
    int ngt = 0, neq = 0;
    for_rows(key, ck, ex, [&](int, uint32_t kv, bool ok) {
      const bool inb = ok && select_bin(kv) == b1;
      ngt += __popc(__ballot_sync(0xffffffffu, inb && kv > T));
      neq += __popc(__ballot_sync(0xffffffffu, inb && kv == T));
    });
    if (lane == 0) {
      sh.wgt[warp] += ngt;
      sh.weq[warp] = neq;
    }
  }
  __syncthreads();
  warp_prefixes(sh);

  // ---- ordered write over every key
  int o = sh.gtb[warp] + min(sh.eqb[warp], need_eq);
  int eq_run = sh.eqb[warp];
  for_rows(key, ck, ex, [&](int i, uint32_t kv, bool ok) {
    const bool isgt = ok && kv > T;
    const bool iseq = ok && kv == T;
    const uint32_t eqm = __ballot_sync(0xffffffffu, iseq);
    const bool sel = isgt || (iseq && eq_run + __popc(eqm & lt) < need_eq);
    const uint32_t selm = __ballot_sync(0xffffffffu, sel);
    if (sel) emit(o + __popc(selm & lt), i);
    o += __popc(selm);
    eq_run += __popc(eqm);
  });
  __syncthreads();
}

// Both tiers of one sequence by the general path (one CTA): the histograms
// are reloaded; a bitmap in the workspace marks the draft tier.
__device__ void select_general(SelShared& sh, const SelectArgs& A, int b, int s_eff, int w0, int nP,
                               int m1, int f, int32_t* out) {
  const int tid = threadIdx.x;
  uint32_t* gbits = A.bits + size_t(b) * A.bits_words;
  const int* gh = A.hist + size_t(b) * 2 * kBins1;
  for (int j = tid; j < 2 * kBins1; j += kThreads) (&sh.h[0][0])[j] = __ldcg(gh + j);
  const int bm0 = s_eff & ~127;
  const int nwords = (w0 - bm0 + 31) / 32;
  for (int j = tid; j < nwords; j += kThreads) gbits[j] = 0u;
  __syncthreads();
  const float* row0 = A.imp + (size_t(b) * 2 + 0) * A.Lcap;
  const float* row1 = A.imp + (size_t(b) * 2 + 1) * A.Lcap;
  const Keys key0{row0, A.err}, key1{row1, A.err};
  if (m1 > 0) {
    const Emit emit{out + nP, m1, f > 0 ? gbits : nullptr, bm0, f > 0 ? &key1 : nullptr, sh.h[1], A.err};
    tier_general(sh, key0, Excl{nullptr, bm0}, s_eff, w0, m1, sh.h[0], emit, A.err);
  }
  if (f > 0) {
    const Emit emit{out + nP + m1, f, nullptr, bm0, nullptr, nullptr, A.err};
    tier_general(sh, key1, Excl{m1 > 0 ? gbits : nullptr, bm0}, s_eff, w0, f, sh.h[1], emit, A.err);
  }
}

// ------------------------------------------------------------ fast finish

// Block-wide exclusive prefixes of two per-thread counts (in place).
__device__ void block_prefix2(SelShared& sh, int& a, int& b) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, ia, o);
    const int z = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += y;
      ib += z;
    }
  }
  if (lane == 31) {
    sh.wgt[warp] = ia;
    sh.weq[warp] = ib;
  }
  __syncthreads();
  warp_prefixes(sh);   // gtb, eqb: exclusive prefixes over the warps
  a = sh.gtb[warp] + ia - a;
  b = sh.eqb[warp] + ib - b;
}

// Exact top cnt of the gathered entries key/pos[0..n) (in position order),
// minus the entries marked in dropbits (if given), given the tier's level-1
// bin b1 and how many of its keys are taken (need): written in position order
// to out[0..cnt); with sub (the target keys of the entries), each selected
// entry's target key is taken out of h1.  With record (the draft tier), the
// exact threshold key goes to sh.t_draft and the last position taken at that
// key to sh.tie_cut: a position is in the tier iff its key is above the
// threshold, or equal to it at a position up to the cut.  With dkey (the
// target tier), entries in the draft tier are left out by that test.
__device__ void finish_tier(SelShared& sh, const uint32_t* key, const int* pos, int n, uint32_t b1,
                            int need, int cnt, int32_t* out, bool record, const uint32_t* dkey,
                            const uint32_t* sub, int* h1) {
  // with dkey (the draft keys of the entries), an entry the draft tier took
  // is left out: its draft key is above that tier's threshold, or equal to it
  // at a position up to the tier's tie cut
  const uint32_t T0 = sh.t_draft;
  const int cut = sh.tie_cut;
  auto drop = [&](int j) {
    if (!dkey) return false;
    const uint32_t k0 = dkey[j];
    return k0 > T0 || (k0 == T0 && pos[j] <= cut);
  };
  const int tid = threadIdx.x;
  const uint32_t T = refine(sh, b1, &need, [&](auto f) {
    for (int j = tid; j < n; j += kThreads) {
      const uint32_t kv = key[j];
      f(kv, select_bin(kv) == b1 && !drop(j));
    }
  });
  const int need_eq = need;
  // one contiguous run of entries per thread, in order
  const int q = (n + kThreads - 1) / kThreads;
  const int j0 = min(n, tid * q), j1 = min(n, j0 + q);
  int ngt = 0, neq = 0;
  for (int j = j0; j < j1; ++j) {
    if (drop(j)) continue;
    const uint32_t kv = key[j];
    ngt += kv > T;
    neq += kv == T;
  }
  block_prefix2(sh, ngt, neq);
  int o = ngt + min(neq, need_eq);
  int eq_run = neq;
  for (int j = j0; j < j1; ++j) {
    if (drop(j)) continue;
    const uint32_t kv = key[j];
    bool sel = kv > T;
    if (kv == T) {
      sel = eq_run++ < need_eq;
      if (sel && record) atomicMax(&sh.tie_cut, pos[j]);
    }
    if (sel) {
      if (o < cnt) out[o] = pos[j];
      if (sub) atomicSub(&h1[select_bin(sub[j])], 1);
      ++o;
    }
  }
  if (record && tid == 0) sh.t_draft = T;
  __syncthreads();
}

// ------------------------------------------------------------------ kernels

__global__ void __launch_bounds__(kThreads, 1) select_kernel(const __grid_constant__ SelectArgs A) {
  extern __shared__ __align__(16) unsigned char dsm[];
  SelShared& sh = *reinterpret_cast<SelShared*>(dsm);
  pdl_launch_dependents();
  pdl_wait();
  cg::cluster_group cluster = cg::this_cluster();
  const int CS = A.cs;   // the cluster size
  const int b = blockIdx.x / CS, r = int(cluster.block_rank());
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lt = (1u << lane) - 1u;
  int32_t* out = A.out + size_t(b) * A.k;
  // the level-1 histograms: their loads go out with the length's
  const int* gh = A.hist + size_t(b) * 2 * kBins1;
  constexpr int kHpt = 2 * kBins1 / kThreads;   // histogram words per thread
  int hv[kHpt];
#pragma unroll
  for (int u = 0; u < kHpt; ++u) hv[u] = __ldcg(gh + tid + u * kThreads);
  const int L = A.seq_len[b];
  // the early cases depend on the sequence only: all its CTAs leave together
  if (L < 0 || L > A.Lcap) {
    if (r == 0) {
      if (tid == 0) flag_error(A.err, DUSTIN_DEV_SEQLEN);
      for (int j = tid; j < A.k; j += kThreads) out[j] = -1;
    }
    return;
  }
  if (A.k >= L) {
    if (r == 0)
      for (int j = tid; j < A.k; j += kThreads) out[j] = j < L ? j : -1;
    return;
  }
  const int s_eff = min(A.sinks, L);
  const int w0 = max(L - A.window, s_eff);
  const int nP = s_eff + (L - w0);
  const int m1 = min(A.m, A.k - nP);
  const int f = A.k - nP - m1;
  if (r == 0)
    for (int j = tid; j < nP; j += kThreads) out[j] = j < s_eff ? j : w0 + (j - s_eff);

  // this CTA's run of U, whole 128-position rows per warp; the first row's
  // keys are loaded now, so that they arrive during the threshold search
  const int a0 = s_eff & ~127;
  const int span = ((((w0 - a0) + CS - 1) / CS) + 127) & ~127;
  const int c0 = a0 + r * span, c1 = min(c0 + span, w0);
  const int wspan = c1 > c0 ? ((((c1 - c0) + kWarps - 1) / kWarps) + 127) & ~127 : 128;
  const int x0 = c0 + warp * wspan, x1 = min(x0 + wspan, c1);
  const float* row0 = A.imp + (size_t(b) * 2 + 0) * A.Lcap;
  const float* row1 = A.imp + (size_t(b) * 2 + 1) * A.Lcap;
  bool have_pre = A.vec4 && x0 < x1;
  float4 pre[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  if (have_pre && x0 + 4 * lane < x1) {
    pre[0] = __ldg(reinterpret_cast<const float4*>(row0 + x0 + 4 * lane));
    pre[1] = __ldg(reinterpret_cast<const float4*>(row1 + x0 + 4 * lane));
  }

  // ---- scan: thresholds from the histograms
#pragma unroll
  for (int u = 0; u < kHpt; ++u) (&sh.h[0][0])[tid + u * kThreads] = hv[u];
  if (tid == 0) {
    sh.overflow = 0;
    sh.tie_cut = -1;
    sh.t_draft = 0xFFFFFFFFu;
  }
  __syncthreads();
  uint32_t b0 = 0xFFFFFFFFu, b1 = 0xFFFFFFFFu;   // no key reaches these bins
  int need0 = 0, need1 = 0;
  long long est = 0;   // entries of the lists of whole threshold bins
  find_bin2(sh, sh.h[0], m1, sh.h[1], f > 0 ? m1 + f : 0);
  if (m1 > 0) {
    if (sh.found2[0]) {
      b0 = uint32_t(sh.bin2[0]);
      need0 = sh.need2[0];
      est += m1 - need0 + sh.h[0][b0];
    } else if (tid == 0) {
      sh.overflow = 1;
    }
  }
  if (f > 0) {
    if (sh.found2[1]) {
      b1 = uint32_t(sh.bin2[1]);
      need1 = sh.need2[1];
      est += m1 + f - need1 + sh.h[1][b1];
    } else if (tid == 0) {
      sh.overflow = 1;
    }
  }
  // list thresholds as keys (0xFFFFFFFF: nothing listed)
  uint32_t t0 = b0 == 0xFFFFFFFFu ? 0xFFFFFFFFu : b0 << 20;
  uint32_t t1 = b1 == 0xFFFFFFFFu ? 0xFFFFFFFFu : b1 << 20;

  // ---- scan of this CTA's run
  bool bad = false;
  // f(i0, kv): every 128-position row of this warp's run, lane holding keys
  // i0 .. i0 + 3 of both channels (0 outside U or past the run)
  auto for_rows4 = [&](auto f) {
    for (int gb = x0; gb < x1; gb += 128) {
      const int i0 = gb + 4 * lane;
      float v[2][4];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const float* row = c ? row1 : row0;
        if (have_pre) {   // the first row, loaded before the threshold search
          const float4 x = pre[c];
          v[c][0] = x.x;
          v[c][1] = x.y;
          v[c][2] = x.z;
          v[c][3] = x.w;
        } else if (A.vec4) {
          const float4 x = i0 < x1 ? __ldg(reinterpret_cast<const float4*>(row + i0)) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[c][0] = x.x;
          v[c][1] = x.y;
          v[c][2] = x.z;
          v[c][3] = x.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) v[c][e] = i0 + e < x1 ? __ldg(row + i0 + e) : 0.f;
        }
      }
      have_pre = false;
      uint32_t kv[2][4];
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = i0 + e;
          const bool ok = i >= s_eff && i < x1;
          const uint32_t bits = __float_as_uint(v[c][e]);
          bad |= ok && bits > 0x7F800000u && bits != 0x80000000u;
          kv[c][e] = (ok && bits <= 0x7F800000u) ? bits : 0u;   // importance_key; flag raised once below
        }
      f(i0, kv);
    }
  };

  // ---- narrower list thresholds when whole bins would not fit (see above)
  if (est > kFinCap) {
    for (int j = tid; j < 2 * kBins2; j += kThreads) (&sh.u.r2[0][0])[j] = 0;
    __syncthreads();
    for_rows4([&](int, const uint32_t (&kv)[2][4]) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint32_t bb = c ? b1 : b0;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          hist_add(sh.u.r2[c], (kv[c][e] >> 10) & 1023u, select_bin(kv[c][e]) == bb && kv[c][e] != 0u,
                   lane);
      }
    });
    cluster.sync();   // every rank's sub-bin histograms are complete
    if (r == 0) {
      int* sum = reinterpret_cast<int*>(sh.ekey);   // [2][kBins2], free until the hand-off
      for (int j = tid; j < 2 * kBins2; j += kThreads) {
        int acc = 0;
        for (int rr = 0; rr < CS; ++rr) acc += (&cluster.map_shared_rank(&sh, rr)->u.r2[0][0])[j];
        sum[j] = acc;
      }
      __syncthreads();
      uint32_t thr0 = t0, thr1 = t1;
      if (b0 != 0xFFFFFFFFu) {
        find_bin(sh, sum, kBins2, need0);
        if (sh.found) thr0 = (b0 << 20) | (uint32_t(sh.bin) << 10);
      }
      if (b1 != 0xFFFFFFFFu) {
        find_bin(sh, sum + kBins2, kBins2, need1);
        if (sh.found) thr1 = (b1 << 20) | (uint32_t(sh.bin) << 10);
      }
      if (tid == 0) {
        sh.thr[0] = thr0;
        sh.thr[1] = thr1;
      }
    }
    cluster.sync();   // rank 0's thresholds are set; every histogram has been read
    const SelShared* r0 = cluster.map_shared_rank(&sh, 0);
    t0 = r0->thr[0];
    t1 = r0->thr[1];
  }

  if (est <= kFinCap) cluster_arrive_relaxed();   // waited for before the hand-off

  // ---- scan: the lists
  int n0 = 0, n1 = 0;   // list entries of this warp (warp-uniform)
  for_rows4([&](int i0, const uint32_t (&kv)[2][4]) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint32_t thr = c ? t1 : t0;
      uint32_t m[4];
      int before = 0, total = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool ok = i0 + e >= s_eff && i0 + e < x1;
        m[e] = __ballot_sync(0xffffffffu, ok && kv[c][e] >= thr);
        before += __popc(m[e] & lt);
        total += __popc(m[e]);
      }
      if (total == 0) continue;   // warp-uniform: nothing of this row is listed
      int& n = c ? n1 : n0;
      int slot = n + before;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if ((m[e] >> lane) & 1u) {
          if (slot < kListCap) {
            if (c) {
              sh.u.l.k1[warp][slot] = kv[1][e];
              sh.u.l.p1[warp][slot] = i0 + e;
              sh.u.l.k1d[warp][slot] = kv[0][e];
            } else {
              sh.u.l.k0[warp][slot] = kv[0][e];
              sh.u.l.k0t[warp][slot] = kv[1][e];
              sh.u.l.p0[warp][slot] = i0 + e;
            }
          }
          ++slot;
        }
      }
      n += total;
    }
  });
  if (__any_sync(0xffffffffu, bad) && lane == 0) flag_error(A.err, DUSTIN_DEV_NAN);
  // ---- hand-off: every warp's list counts (and whether its lists or the
  // threshold search overflowed) go to every rank; after a cluster barrier
  // each rank derives every list's offset and pushes its entries into rank
  // 0's arrays, in position order; a second barrier completes them
  if (est <= kFinCap) cluster_wait();   // every CTA of the cluster has started
  if (lane == 0) {
    const int ovf = (n0 > kListCap || n1 > kListCap || sh.overflow) ? 1 : 0;
    for (int rr = 0; rr < CS; ++rr) {
      SelShared* rs = cluster.map_shared_rank(&sh, rr);
      rs->cell[0][r * kWarps + warp] = min(n0, kListCap);
      rs->cell[1][r * kWarps + warp] = min(n1, kListCap);
      rs->ovf_all[r * kWarps + warp] = ovf;
    }
  }
  cluster.sync();
  if (tid < 2 * 32) {   // exclusive prefix over the CS * 32 cells of each channel
    const int c = tid >> 5, lane2 = tid & 31;
    int carry = 0;
    for (int base = 0; base < CS * kWarps; base += 32) {
      const int v = sh.cell[c][base + lane2];
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane2 >= o) incl += y;
      }
      sh.cell[c][base + lane2] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane2 == 0) sh.cell[c][CS * kWarps] = carry;
  } else if (tid < 3 * 32) {   // any overflow anywhere
    int o = 0;
    for (int i = lane; i < CS * kWarps; i += 32) o |= sh.ovf_all[i];
    o = __any_sync(0xffffffffu, o != 0);
    if (lane == 0) sh.overflow = o;
  }
  __syncthreads();
  const int n0t = sh.cell[0][CS * kWarps], n1t = sh.cell[1][CS * kWarps];
  if (!sh.overflow && n0t + n1t <= kFinCap) {
    SelShared* r0 = cluster.map_shared_rank(&sh, 0);
    const int base0 = sh.cell[0][r * kWarps + warp], base1 = n0t + sh.cell[1][r * kWarps + warp];
    for (int slot = lane; slot < n0; slot += 32) {
      r0->ekey[base0 + slot] = sh.u.l.k0[warp][slot];
      r0->ek0t[base0 + slot] = sh.u.l.k0t[warp][slot];
      r0->epos[base0 + slot] = sh.u.l.p0[warp][slot];
    }
    for (int slot = lane; slot < n1; slot += 32) {
      r0->ekey[base1 + slot] = sh.u.l.k1[warp][slot];
      r0->ek0t[base1 + slot] = sh.u.l.k1d[warp][slot];
      r0->epos[base1 + slot] = sh.u.l.p1[warp][slot];
    }
  }
  cluster.sync();   // rank 0 holds every entry: the others may leave
  if (r != 0) return;

  // ---- finish (rank 0)
  if (sh.overflow || n0t + n1t > kFinCap) {
    select_general(sh, A, b, s_eff, w0, nP, m1, f, out);
    return;
  }
  if (m1 > 0)
    finish_tier(sh, sh.ekey, sh.epos, n0t, b0, need0, m1, out + nP, f > 0, nullptr,
                f > 0 ? sh.ek0t : nullptr, sh.h[1]);
  if (f > 0) {
    // the target histogram of U minus the draft tier (corrected above), and
    // its threshold bin
    find_bin(sh, sh.h[1], kBins1, f);
    if (!sh.found) {   // cannot happen with matching keys
      if (tid == 0) flag_error(A.err, DUSTIN_DEV_NAN);
      return;
    }
    const uint32_t bt = uint32_t(sh.bin);
    const int needt = sh.need;
    // the target entries the draft tier took are left out by their draft keys
    finish_tier(sh, sh.ekey + n0t, sh.epos + n0t, n1t, bt, needt, f, out + nP + m1, false,
                m1 > 0 ? sh.ek0t + n0t : nullptr, nullptr, nullptr);
  }
}

// Standalone selection: the level-1 histograms of both channels over each
// sequence's unprotected positions (the fused step builds them while scoring).
__global__ void __launch_bounds__(kHistThreads) select_hist_kernel(const __grid_constant__ SelectArgs A) {
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.y;
  const int i = blockIdx.x * kHistThreads + threadIdx.x;
  const int lane = threadIdx.x & 31;
  int L = A.seq_len[b];
  if (L < 0 || L > A.Lcap) L = 0;
  const int s_eff = min(A.sinks, L);
  const int w0 = max(L - A.window, s_eff);
  const bool in_u = i >= s_eff && i < w0;
  int* h = A.hist + size_t(b) * 2 * kBins1;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t kv = in_u ? importance_key(A.imp[(size_t(b) * 2 + c) * A.Lcap + i], A.err) : 0u;
    hist_add(h + c * kBins1, select_bin(kv), in_u, lane);
  }
}

}  // namespace

namespace {

// How many clusters of cs select CTAs can be resident at once on the current
// device (cached per device and cluster size).
int max_active_clusters(int cs) {
  struct Entry {
    int dev, cs, n;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.dev == dev && e.cs == cs) return e.n;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(cs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(SelShared);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cs;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sizeof(SelShared))) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, select_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache.push_back({dev, cs, n});
  return n;
}

}  // namespace

int select_ctas_per_sequence(int B) {
  // the largest cluster (8, 4 or 2 CTAs) whose B clusters are all resident at
  // once and that keeps the scan to about 128 CTAs; one CTA per sequence when
  // even pairs do not fit
  for (int cs = kMaxSelectCtas; cs >= 2; cs >>= 1)
    if ((long long)B * cs <= 128 && B <= max_active_clusters(cs)) return cs;
  return 1;
}

SelectPlan select_plan(int B, int Lcap, size_t off) {
  SelectPlan s{};
  s.bits_words = (Lcap + 127) / 32 + 2;
  auto r256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  s.hist_off = off;
  s.bits_off = s.hist_off + r256(size_t(B) * 2 * kBins1 * 4);
  s.end = s.bits_off + r256(size_t(B) * s.bits_words * 4);
  return s;
}

cudaError_t select_launch(const SelectArgs& a0, bool build_hist, cudaStream_t stream) {
  SelectArgs a = a0;
  a.cs = select_ctas_per_sequence(a.B);
  a.vec4 = (a.Lcap % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.imp) & 15u) == 0);
  cudaError_t e;
  if (build_hist) {
    if ((e = cudaMemsetAsync(a.hist, 0, size_t(a.B) * 2 * kBins1 * 4, stream)) != cudaSuccess) return e;
    e = launch_pdl(select_hist_kernel, dim3((a.Lcap + kHistThreads - 1) / kHistThreads, a.B),
                   dim3(kHistThreads), 0, stream, a);
    if (e != cudaSuccess) return e;
  }
  const size_t smem = sizeof(SelShared);
  static const cudaError_t attr =
      cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.B * a.cs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = a.cs;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, select_kernel, a);
}

}  // namespace dustin
