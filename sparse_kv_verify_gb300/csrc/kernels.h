// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/dustin.h"

namespace dustin {

// ------------------------------------------------------------------ verify

struct VerifyLayerDev {
  const uint16_t* q;   // [B][T][hq][D]
  const uint16_t* k;   // cache base
  const uint16_t* v;
  const uint16_t* kb;  // [B][hkv][T][D]
  const uint16_t* vb;
  float* o;            // [B][T][hq][D]
  int64_t ksb, ksh, ksl, vsb, vsh, vsl;
};

struct VerifyArgs {
  int B, Lcap, T, hq, hkv, G, NQ;
  int k;                // budget (sparse); unused for dense
  int dense;            // 1: keys are positions 0..seq_len-1
  int keys_per_split;   // multiple of 64
  int n_layers;
  float scale_log2;     // log2(e) / sqrt(D)
  const int32_t* ivf;   // [B][k] (sparse)
  const int32_t* seq_len;
  int* err;
  VerifyLayerDev layer[DUSTIN_MAX_LAYERS];
};

struct VerifyLaunch {
  int D, MT, NST, CS;
  size_t smem;
};

VerifyLaunch verify_plan(int D, int NQ, int nkeys_cap, int B, int hkv, int n_layers, int dense);
cudaError_t verify_launch(const VerifyArgs& a, const VerifyLaunch& pl, cudaStream_t stream);

// ------------------------------------------------------------------- score

struct ScoreSlab {
  int channel;   // 0 draft, 1 target
  int cache;     // index into ScoreArgs::map
  int g;         // KV head
  int D;         // head dim (64 or 128)
  int nq;        // query rows per sequence
  int hq;        // query heads of the model
  int npairs;    // heads.size() * nq
  int nheads;
  int heads[DUSTIN_MAX_PAIRS];
  const uint16_t* q;  // [B][nq][hq][D]
};

struct ScoreArgs {
  CUtensorMap map[DUSTIN_MAX_SRH];   // one per (channel, layer) cache
  ScoreSlab slab[DUSTIN_MAX_SRH];
  int B, Lcap, C, P, LS, n_slab, np_max;
  const int32_t* seq_len;
  int* err;
  float* part;          // [n_slab][B][Lcap]
  float* spill;         // logits in global memory when they do not fit on chip
};

struct ScoreLaunch {
  int C, P, LS, NT, np_max;
  bool smem_logits;
  size_t smem;
  size_t spill_bytes;
};

ScoreLaunch score_plan(int Lcap, int B, int n_slab, int np_max, int d_max);
cudaError_t score_launch(const ScoreArgs& a, const ScoreLaunch& pl, cudaStream_t stream);

struct ReduceArgs {
  int B, Lcap, n_slab;
  int channel_of[DUSTIN_MAX_SRH];
  const float* part;
  const int32_t* seq_len;
  float* importance;   // [B][2][Lcap]
};
cudaError_t score_reduce_launch(const ReduceArgs& a, cudaStream_t stream);

// ------------------------------------------------------------------ select

struct SelectArgs {
  int B, Lcap, k, sinks, window, m;
  int cache_keys;        // 1: stage keys in shared memory
  const float* imp;      // [B][2][Lcap]
  const int32_t* seq_len;
  int32_t* out;          // [B][k]
  int* err;
};
size_t select_smem_bytes(int Lcap, int cache_keys);
int select_cache_keys(int Lcap);
cudaError_t select_launch(const SelectArgs& a, cudaStream_t stream);

// ------------------------------------------------------------------ append

struct AppendLayerDev {
  uint16_t* k;
  uint16_t* v;
  const uint16_t* kb;
  const uint16_t* vb;
  int64_t ksb, ksh, ksl, vsb, vsh, vsl;
};

struct AppendArgs {
  int B, Lcap, T, hkv, D, n_layers;
  const int32_t* n_accept;
  int32_t* seq_len;
  int* err;
  AppendLayerDev layer[DUSTIN_MAX_LAYERS];
};
cudaError_t append_launch(const AppendArgs& a, cudaStream_t stream);

}  // namespace dustin
