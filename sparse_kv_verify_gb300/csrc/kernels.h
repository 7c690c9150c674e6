// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/dustin.h"

namespace dustin {

// Launches kern<<<grid, block, smem, stream>>>(args) with programmatic stream
// serialisation, so that it may begin while the previous kernel in the stream
// drains (the kernel itself waits with pdl_wait before reading its inputs).
template <typename Kern, typename Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       const Args& args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

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

// Shared-memory layout of the verification kernel (bytes from its 1024-byte
// aligned base), chosen on the host per launch.
struct VLay {
  int NP, nst;           // 64-column panels per row; K/V stages
  uint32_t q_panel, q_buf, ring_off, kv_panel, half_bytes, stage_bytes;
  uint32_t mask_off, bar_off, misc_off, total;
};

struct VerifyArgs {
  int B, Lcap, T, hq, hkv, G, NQ;
  int k;                // budget (sparse); unused for dense
  int dense;            // 1: keys are positions 0..seq_len-1
  int n_layers;
  int ctx_tiles;        // 64-key tiles of context per unit
  int tiles_u;          // ctx_tiles + 1 (the draft-block tile)
  long long total;      // units * tiles_u
  int max_seg;          // partial slots per unit
  long long slot_floats;  // floats per partial slot (multiple of 4)
  float scale_log2;     // log2(e) / sqrt(D)
  VLay lay;
  const int32_t* ivf;   // [B][k] (sparse)
  const int32_t* seq_len;
  int* err;
  float* partial;       // [units][max_seg][slot_floats]: O [NQ][D], m [NQ], l [NQ]
  VerifyLayerDev layer[DUSTIN_MAX_LAYERS];
  // per layer: the queries as 3-D (d, hq, B*T) with box (64, G, T) and the
  // 128-byte swizzle, so one load brings a unit's G x T query rows
  CUtensorMap qmap[DUSTIN_MAX_LAYERS];
  // dense mode, tma = 1: per layer the K and V caches as tensor maps with a
  // (64 columns, 64 rows) box and the 128-byte swizzle (rank 2: rows
  // B*hkv*Lcap of a packed cache; rank 4: (d, Lcap, hkv, B) of a strided one),
  // so that a context tile wholly inside the sequence comes in 2 * D / 64
  // boxes instead of row gathers
  int tma;
  int kvrank[DUSTIN_MAX_LAYERS];
  CUtensorMap kmap[DUSTIN_MAX_LAYERS];
  CUtensorMap vmap[DUSTIN_MAX_LAYERS];
};

// The segment merge that follows the stream-K kernel.
struct VerifyCombineArgs {
  int NQ, T, hq, hkv, G, units_per_layer, tiles_u, main_grid, max_seg;
  long long total, slot_floats;
  const float* partial;
  float* o[DUSTIN_MAX_LAYERS];
};

struct VerifyLaunch {
  int D, NST;
  int cps;               // CTAs per SM (1 or 2)
  VLay lay;
  int ctx_tiles, tiles_u, grid, max_seg;
  long long units, total, slot_floats;
  size_t smem;
};

// Grid sizes never exceed kVerifyGridMax, which bounds the partial slots.
constexpr int kVerifyGridMax = 1024;
VerifyLaunch verify_plan(int D, int NQ, int nkeys_cap, int B, int hkv, int n_layers, int dense,
                         int num_sms);
size_t verify_scratch_bytes(const VerifyLaunch& pl);
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
  int rows;      // positions per tile (128 for d = 128, 256 for d = 64)
  int tiles;     // tiles per sequence: ceil(Lcap / rows)
  long long logit_off;   // float offset of this slab's logits [nb][npairs][LSP]
  int row2d;     // 0: 4-D map; else 2-D map over packed rows, value = hkv of the cache
  int cost;      // relative cost of one tile (bytes plus logits written), for balancing
  const uint16_t* q;     // [B][nq][hq][D]
};

// Per-slab facts of one group launch in a compact form: the normalise kernel
// copies the table to shared memory once (kernel-parameter reads with a
// per-thread index are slow) and walks it there.
struct SlabInfo {
  long long logit_off;   // float offset of the slab's logits
  long long first_tile;  // first flattened tile of the slab
  long long cost_start;  // cost before that tile
  int npairs, tiles, cost, row0;   // row0: the slab's first logits row (channel 0 first)
  int slab, pad;         // index of the slab in ScoreArgs::slab
};

// One stream launch as the normalise kernel sees it.
struct NormGroup {
  int b0, nb;            // its sequences
  int grid;              // CTAs of its stream kernel
  int cps;               // normalise CTAs per sequence
  long long total_cost;  // its partition's total cost
  float* logits;         // its logits buffer
  float* stats;          // its statistics buffer
};


struct ScoreArgs {
  CUtensorMap map[DUSTIN_MAX_SRH];   // one per (channel, layer) cache; box 64 x 128
  ScoreSlab slab[DUSTIN_MAX_SRH];
  long long slab_start[DUSTIN_MAX_SRH + 1];   // first flattened tile of each slab
  long long cost_start[DUSTIN_MAX_SRH + 1];   // cost before the first tile of each slab
  long long total;                            // tiles of this group
  long long total_cost;                       // sum of tile costs of this group
  int B, Lcap, LSP, n_slab, np_max;
  int n_rows, n_rows0;   // logits rows (slab, pair) per sequence, channel 0 first; rows of channel 0
  int sinks, window;     // the unprotected range of the selection histograms
  int b0, nb;            // the group of sequences handled by this launch
  int grid;              // CTAs of the stream kernel
  int max_seg;           // statistics slots per (slab, sequence)
  const int32_t* seq_len;
  int* err;
  float* logits;         // scratch, stays in L2 between the two kernels
  float* stats;          // [n_slab][nb][max_seg][np_max][2]
  float* importance;     // [B][2][Lcap]
  int* hist;             // [B][2][4096] selection histograms, or nullptr
  // stream kernel: 0 -- wait for the previous launch before starting; 1 --
  // start at once (the previous launch is the other stream kernel of a pair,
  // writing other buffers) and wait for it only before exiting, so that this
  // launch completes after it
  int wait_at_end;
  // normalise kernel: the groups it covers (one or two stream launches), each
  // with its own logits and statistics buffers and partition
  int n_groups;
  NormGroup ng[2];
  SlabInfo info[2][DUSTIN_MAX_SRH];   // per group, in row order (channel 0 slabs first)
};

struct ScoreLaunch {
  int NT;
  size_t smem;
  size_t norm_smem;      // dynamic shared memory of the normalise kernel
};

constexpr int kScoreGridMax = 256;
size_t score_stream_smem();
size_t score_norm_smem(int n_rows);
int score_norm_ctas_per_sm(int n_rows);   // resident normalise CTAs per SM
int score_rows_per_tile(int D);
int score_tile_cost(int D, int npairs);
// Launches the stream kernel of the group in a (b0, nb, logits, stats, ...).
cudaError_t score_stream_launch(const ScoreArgs& a, const ScoreLaunch& pl, cudaStream_t stream);
// Launches the normalise kernel of the groups in a.ng[0 .. n_groups).
cudaError_t score_norm_launch(const ScoreArgs& a, const ScoreLaunch& pl, cudaStream_t stream);

// ------------------------------------------------------------------ select

constexpr int kMaxSelectCtas = 8;          // scan CTAs (cluster size) per sequence

struct SelectArgs {
  int B, Lcap, k, sinks, window, m;
  int vec4;              // set by select_launch: rows read as float4
  int cs;                // set by select_launch: scan CTAs per sequence (one cluster)
  int bits_words;        // bitmap words per sequence (general path)
  const float* imp;      // [B][2][Lcap]
  int* hist;             // [B][2][4096] level-1 histograms over the unprotected
                         // positions (built by the score kernels in the fused
                         // step, by select_launch otherwise)
  const int32_t* seq_len;
  int32_t* out;          // [B][k]
  int* err;
  uint32_t* bits;        // [B][bits_words]
};

// Workspace layout of the selection scratch starting at byte offset off.
struct SelectPlan {
  int bits_words;
  size_t hist_off, bits_off, end;
};
SelectPlan select_plan(int B, int Lcap, size_t off);
// build_hist: count the histograms first (standalone call).
cudaError_t select_launch(const SelectArgs& a, bool build_hist, cudaStream_t stream);

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

// ----------------------------------------------------------------- compact

struct CompactLayerDev {
  const uint16_t* k;
  const uint16_t* v;
  uint16_t* kc;
  uint16_t* vc;
  int64_t ksb, ksh, ksl, vsb, vsh, vsl;
  int64_t kcsb, kcsh, kcsl, vcsb, vcsh, vcsl;
};

struct CompactArgs {
  int B, Lcap, k, hkv, D, n_layers;
  const int32_t* ivf;        // [B][k]
  const int32_t* seq_len;
  int32_t* seq_len_c;        // [B] out: compact lengths
  int* err;
  CompactLayerDev layer[DUSTIN_MAX_LAYERS];
};
cudaError_t compact_launch(const CompactArgs& a, cudaStream_t stream);

// ------------------------------------------------------------ wait self-test
cudaError_t wait_selftest_launch(int* err, long long* waited, unsigned long long limit_ns,
                                 cudaStream_t stream);

}  // namespace dustin
