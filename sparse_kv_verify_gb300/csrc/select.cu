// Budgeted tiered selection of I_verify ("Technical Summary: Dustin", section
// 1 "Hybrid Attention Aggregation": protect a sink prefix and a local window of
// recent tokens, then fill the rest of the fixed budget with the top-m tokens
// by the draft signal, then the most relevant remaining tokens by the target
// signal).
//
// One 1024-thread CTA per sequence.  Importance values are non-negative fp32,
// so their bit patterns order like the values.  Each tier finds the exact
// threshold key T of its top-cnt (descending key, ties to the lower index):
//   1. a 4096-bin histogram of the top 12 bits (sign, exponent, 3 mantissa
//      bits) of every candidate key -- fine enough that the shared-memory
//      atomics rarely collide -- gives the bin that holds the cnt-th key;
//   2. the keys of that bin are gathered into a small list and two 10-bit
//      radix passes over the list give T and how many keys equal to T to take;
//   3. an order-preserving compaction writes every key > T and the
//      lowest-index keys == T, ascending.
// If the threshold bin holds more keys than the list can take (heavy ties), the
// refinement runs over all candidates instead.  Keys are staged in shared
// memory when the cache capacity allows; the draft tier is recorded in a
// bitmap that the target tier skips.
#include "common.cuh"
#include "kernels.h"

namespace dustin {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins1 = 4096;      // top 12 bits
constexpr int kBins2 = 1024;      // 10 bits
constexpr int kCandCap = 8192;
constexpr size_t kSmemBudget = 200 * 1024;

struct SelShared {
  int hist[kBins1];
  uint32_t cand[kCandCap];
  int wsum[kWarps];
  int wgt[kWarps];
  int weq[kWarps];
  int ncand;
  int bin;
  int need;
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
  const uint32_t* cached;  // shared-memory copy (or nullptr)
  const float* global;     // importance row of this channel
  int* err;
  __device__ __forceinline__ uint32_t operator()(int i) const {
    return cached ? cached[i] : key_of(global[i], err);
  }
};

__device__ __forceinline__ bool excluded(const uint32_t* excl, int i) {
  return excl && ((excl[i >> 5] >> (i & 31)) & 1u);
}

constexpr int kBatch = 8;   // independent key loads in flight per thread

// Calls f(i, key, valid) for every i in [u0, u1), block-strided, with kBatch
// loads issued before any is used (so global-memory keys do not serialise on
// latency).  Every lane of every warp makes the same number of calls.
template <typename F>
__device__ __forceinline__ void for_keys(const KeySrc& key, int u0, int u1, const uint32_t* excl,
                                         F f) {
  for (int base = u0; base < u1; base += kThreads * kBatch) {
    uint32_t kv[kBatch];
    bool ok[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * kThreads + int(threadIdx.x);
      ok[u] = i < u1 && !excluded(excl, i);
      kv[u] = ok[u] ? key(i) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) f(base + u * kThreads + int(threadIdx.x), kv[u], ok[u]);
  }
}

// Over the histogram in descending bin order: the bin holding the need-th key
// and how many keys of that bin are still needed.  Whole-block call.
__device__ void find_bin(SelShared& sh, int nbins, int need) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = nbins / kThreads;   // bins per thread (4 or 1)
  int local = 0;
  for (int k = 0; k < q; ++k) local += sh.hist[nbins - 1 - (tid * q + k)];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = sh.wsum[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    sh.wsum[lane] = wi - w;   // exclusive prefix of the warp sums
  }
  __syncthreads();
  const int before = sh.wsum[warp] + incl - local;
  if (before < need && need <= before + local) {
    int acc = before;
    for (int k = 0; k < q; ++k) {
      const int bin = nbins - 1 - (tid * q + k);
      const int h = sh.hist[bin];
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

// Top `cnt` candidates of [u0, u1) minus `excl` by (key desc, index asc):
// written ascending to out[0..cnt), bits set in `setbits` when given.
__device__ void tier_select(const KeySrc& key, int u0, int u1, const uint32_t* excl, int cnt,
                            int32_t* out, uint32_t* setbits, SelShared& sh) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (cnt <= 0 || u1 <= u0) return;

  // 1. top-12-bit histogram
  for (int b = tid; b < kBins1; b += kThreads) sh.hist[b] = 0;
  if (tid == 0) sh.ncand = 0;
  __syncthreads();
  for_keys(key, u0, u1, excl, [&](int, uint32_t kv, bool ok) {
    if (ok) atomicAdd(&sh.hist[kv >> 20], 1);
  });
  __syncthreads();
  find_bin(sh, kBins1, cnt);
  const uint32_t b1 = uint32_t(sh.bin);
  int need = sh.need;

  // 2. gather the keys of the threshold bin (one atomic per warp)
  for_keys(key, u0, u1, excl, [&](int, uint32_t kv, bool ok) {
    const bool hit = ok && (kv >> 20) == b1;
    const uint32_t ball = __ballot_sync(0xffffffffu, hit);
    if (ball) {
      int slot0 = 0;
      if (lane == 0) slot0 = atomicAdd(&sh.ncand, __popc(ball));
      slot0 = __shfl_sync(0xffffffffu, slot0, 0);
      const int slot = slot0 + __popc(ball & ((1u << lane) - 1u));
      if (hit && slot < kCandCap) sh.cand[slot] = kv;
    }
  });
  __syncthreads();
  const int ncand = sh.ncand;
  const bool listed = ncand <= kCandCap;
  uint32_t prefix = b1 << 20;
  // two 10-bit passes over the list (or over all candidates when it overflowed)
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = 10 - 10 * pass;
    const uint32_t hi_mask = 0xFFFFFFFFu << (shift + 10);
    __syncthreads();
    for (int b = tid; b < kBins2; b += kThreads) sh.hist[b] = 0;
    __syncthreads();
    if (listed) {
      for (int c = tid; c < ncand; c += kThreads) {
        const uint32_t kv = sh.cand[c];
        if ((kv & hi_mask) == prefix) atomicAdd(&sh.hist[(kv >> shift) & 1023u], 1);
      }
    } else {
      for_keys(key, u0, u1, excl, [&](int, uint32_t kv, bool ok) {
        if (ok && (kv & hi_mask) == prefix) atomicAdd(&sh.hist[(kv >> shift) & 1023u], 1);
      });
    }
    __syncthreads();
    find_bin(sh, kBins2, need);
    prefix |= uint32_t(sh.bin) << shift;
    need = sh.need;
  }
  const uint32_t T = prefix;

  // 3. order-preserving compaction over 32-aligned warp chunks
  const int a0 = u0 & ~31;
  const int span = u1 - a0;
  const int chunk = (((span + kWarps - 1) / kWarps) + 31) & ~31;
  const int w0 = a0 + warp * chunk;
  const int w1 = min(w0 + chunk, u1);
  int ngt = 0, neq = 0;
  for (int gb = w0; gb < w1; gb += 32 * kBatch) {
    uint32_t kv[kBatch];
    bool cv[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = gb + 32 * u + lane;
      cv[u] = i >= u0 && i < w1 && !excluded(excl, i);
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
  int gt_before = 0, eq_before = 0;
  for (int w = 0; w < warp; ++w) {
    gt_before += sh.wgt[w];
    eq_before += sh.weq[w];
  }
  int pos = gt_before + min(eq_before, need);
  int eq_run = eq_before;
  const uint32_t lt = (1u << lane) - 1u;
  for (int gb = w0; gb < w1; gb += 32 * kBatch) {
    uint32_t kv[kBatch];
    bool cv[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = gb + 32 * u + lane;
      cv[u] = i >= u0 && i < w1 && !excluded(excl, i);
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
      if (sel) out[pos + __popc(selb & lt)] = i;
      if (setbits && lane == 0 && g0 < w1) setbits[g0 >> 5] |= selb;
      pos += __popc(selb);
      eq_run += __popc(eqb);
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1) select_kernel(const __grid_constant__ SelectArgs A) {
  extern __shared__ __align__(16) unsigned char dsm[];
  SelShared& sh = *reinterpret_cast<SelShared*>(dsm);
  unsigned char* rest = dsm + ((sizeof(SelShared) + 15) & ~size_t(15));
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  int32_t* out = A.out + size_t(b) * A.k;
  const int L = A.seq_len[b];
  if (L < 0 || L > A.Lcap) {
    if (tid == 0) flag_error(A.err, DUSTIN_DEV_SEQLEN);
    for (int j = tid; j < A.k; j += kThreads) out[j] = -1;
    return;
  }
  if (A.k >= L) {
    for (int j = tid; j < A.k; j += kThreads) out[j] = j < L ? j : -1;
    return;
  }
  const int s_eff = min(A.sinks, L);
  const int w0 = max(L - A.window, s_eff);
  const int nP = s_eff + (L - w0);
  const int m1 = min(A.m, A.k - nP);
  const int f = A.k - nP - m1;
  for (int j = tid; j < nP; j += kThreads) out[j] = j < s_eff ? j : w0 + (j - s_eff);

  const int nwords = (A.Lcap + 31) >> 5;
  uint32_t* keys = A.cache_keys ? reinterpret_cast<uint32_t*>(rest) : nullptr;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(rest + (A.cache_keys ? size_t(A.Lcap) * 4 : 0));
  for (int w = tid; w < nwords; w += kThreads) bitmap[w] = 0u;

  for (int ch = 0; ch < 2; ++ch) {
    const float* row = A.imp + (size_t(b) * 2 + ch) * A.Lcap;
    if (keys) {
      for (int base = s_eff; base < w0; base += kThreads * kBatch) {
        float v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int i = base + u * kThreads + tid;
          v[u] = i < w0 ? row[i] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int i = base + u * kThreads + tid;
          if (i < w0) keys[i] = key_of(v[u], A.err);
        }
      }
    }
    __syncthreads();
    KeySrc src{keys, row, A.err};
    if (ch == 0) tier_select(src, s_eff, w0, nullptr, m1, out + nP, bitmap, sh);
    else tier_select(src, s_eff, w0, bitmap, f, out + nP + m1, nullptr, sh);
    __syncthreads();
  }
}

}  // namespace

int select_cache_keys(int Lcap) {
  const size_t need = sizeof(SelShared) + 16 + size_t(Lcap) * 4 + size_t((Lcap + 31) / 32) * 4;
  return need <= kSmemBudget ? 1 : 0;
}

size_t select_smem_bytes(int Lcap, int cache_keys) {
  return ((sizeof(SelShared) + 15) & ~size_t(15)) + (cache_keys ? size_t(Lcap) * 4 : 0) +
         size_t((Lcap + 31) / 32) * 4;
}

cudaError_t select_launch(const SelectArgs& a, cudaStream_t stream) {
  const size_t smem = select_smem_bytes(a.Lcap, a.cache_keys);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(select_kernel, dim3(a.B), dim3(kThreads), smem, stream, a);
}

}  // namespace dustin
