// Budgeted tiered selection of I_verify ("Technical Summary: Dustin", section
// 1 "Hybrid Attention Aggregation": protect a sink prefix and a local window of
// recent tokens, then fill the rest of the fixed budget with the top-m tokens
// by the draft signal, then the most relevant remaining tokens by the target
// signal).
//
// One 1024-thread CTA per sequence.  Importance values are non-negative fp32,
// so their bit patterns order like the values; each tier is a radix select of
// the threshold key T over four 8-bit digits (per-digit histograms built with
// warp-aggregated shared-memory atomics), followed by an order-preserving
// compaction that takes every key > T and the lowest-index keys == T until the
// tier is full.  Keys are staged in shared memory when the cache capacity
// allows; the draft tier is recorded in a bitmap that the target tier skips.
#include "common.cuh"
#include "kernels.h"

namespace dustin {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr size_t kSmemBudget = 200 * 1024;

struct SelShared {
  int hist[256];
  int wgt[kWarps];
  int weq[kWarps];
  int digit;
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

// Selects the top `cnt` candidates of [u0, u1) (minus bits set in `excl`) by
// (key descending, index ascending), writes them ascending to out[0..cnt) and
// sets their bits in `setbits` when given.  Whole-block call.
__device__ void tier_select(const KeySrc& key, int u0, int u1, const uint32_t* excl, int cnt,
                            int32_t* out, uint32_t* setbits, SelShared& sh) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (cnt <= 0 || u1 <= u0) return;
  uint32_t prefix = 0, pmask = 0;
  int need = cnt;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (tid < 256) sh.hist[tid] = 0;
    __syncthreads();
    for (int base = u0; base < u1; base += kThreads) {
      const int i = base + tid;
      bool c = i < u1 && !(excl && ((excl[i >> 5] >> (i & 31)) & 1u));
      uint32_t kv = 0;
      if (c) {
        kv = key(i);
        c = (kv & pmask) == prefix;
      }
      const uint32_t dg = c ? ((kv >> shift) & 255u) : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, dg);
      if (c && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[dg], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      // lane l covers digits 255-8l down to 248-8l
      int cnt8[8];
      int local = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        cnt8[q] = sh.hist[255 - 8 * lane - q];
        local += cnt8[q];
      }
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int before = incl - local;
      if (before < need && need <= incl) {
        int acc = before;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (acc + cnt8[q] >= need) {
            sh.digit = 255 - 8 * lane - q;
            sh.need = need - acc;
            break;
          }
          acc += cnt8[q];
        }
      }
    }
    __syncthreads();
    prefix |= uint32_t(sh.digit) << shift;
    pmask |= 255u << shift;
    need = sh.need;
    __syncthreads();
  }
  const uint32_t T = prefix;

  // order-preserving compaction over 32-aligned warp chunks
  const int a0 = u0 & ~31;
  const int span = u1 - a0;
  const int chunk = (((span + kWarps - 1) / kWarps) + 31) & ~31;
  const int w0 = a0 + warp * chunk;
  const int w1 = min(w0 + chunk, u1);
  int ngt = 0, neq = 0;
  for (int g0 = w0; g0 < w1; g0 += 32) {
    const int i = g0 + lane;
    bool c = i >= u0 && i < w1 && !(excl && ((excl[i >> 5] >> (i & 31)) & 1u));
    uint32_t kv = c ? key(i) : 0u;
    ngt += __popc(__ballot_sync(0xffffffffu, c && kv > T));
    neq += __popc(__ballot_sync(0xffffffffu, c && kv == T));
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
  for (int g0 = w0; g0 < w1; g0 += 32) {
    const int i = g0 + lane;
    bool c = i >= u0 && i < w1 && !(excl && ((excl[i >> 5] >> (i & 31)) & 1u));
    uint32_t kv = c ? key(i) : 0u;
    const bool isgt = c && kv > T;
    const bool iseq = c && kv == T;
    const uint32_t eqb = __ballot_sync(0xffffffffu, iseq);
    const bool sel = isgt || (iseq && (eq_run + __popc(eqb & lt)) < need);
    const uint32_t selb = __ballot_sync(0xffffffffu, sel);
    if (sel) out[pos + __popc(selb & lt)] = i;
    if (setbits && lane == 0) setbits[g0 >> 5] |= selb;
    pos += __popc(selb);
    eq_run += __popc(eqb);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1) select_kernel(const __grid_constant__ SelectArgs A) {
  __shared__ SelShared sh;
  extern __shared__ __align__(16) unsigned char dsm[];
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
  uint32_t* keys = A.cache_keys ? reinterpret_cast<uint32_t*>(dsm) : nullptr;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(dsm + (A.cache_keys ? size_t(A.Lcap) * 4 : 0));
  for (int w = tid; w < nwords; w += kThreads) bitmap[w] = 0u;

  for (int ch = 0; ch < 2; ++ch) {
    const float* row = A.imp + (size_t(b) * 2 + ch) * A.Lcap;
    if (keys) {
      for (int i = s_eff + tid; i < w0; i += kThreads) keys[i] = key_of(row[i], A.err);
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
  const size_t need = size_t(Lcap) * 4 + size_t((Lcap + 31) / 32) * 4;
  return need <= kSmemBudget ? 1 : 0;
}

size_t select_smem_bytes(int Lcap, int cache_keys) {
  return (cache_keys ? size_t(Lcap) * 4 : 0) + size_t((Lcap + 31) / 32) * 4;
}

cudaError_t select_launch(const SelectArgs& a, cudaStream_t stream) {
  const size_t smem = select_smem_bytes(a.Lcap, a.cache_keys);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(smem));
  if (e != cudaSuccess) return e;
  select_kernel<<<a.B, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dustin
