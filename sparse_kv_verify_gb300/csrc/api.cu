// C-ABI layer: argument validation, launch planning, TMA descriptor encoding
// and kernel launches for the calls declared in include/dustin.h.  Nothing
// here allocates device memory; scratch lives in the caller's workspace:
//   [0, 256)                 header: the sticky device error word (int32 at 0)
//   [256, 256 + 64 KiB)      reserved (cleared by dustin_workspace_init)
//   [kScratch, ...)          scratch shared by the stages of one call:
//                            score: logits of one group of sequences
//                                   [n_slab][nb][pairs][LSP] (kept in L2) and
//                                   per-segment (max, sum) statistics
//                            select (after the score scratch in the fused
//                                   step): histograms, bitmaps
//                            verify: segment partials [units][max_seg][slot]
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

using namespace dustin;

namespace {

constexpr size_t kHeader = 256;
constexpr size_t kCounterBytes = 65536;   // reserved
constexpr long long kVerifyUnitsMax = 16384;        // B * Hkv * layers per verification call
constexpr size_t kScratch = kHeader + kCounterBytes;

int num_sms() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool params_ok(const dustin_params* p) {
  if (!p) return false;
  if (p->B < 1 || p->B > 65535) return false;
  if (p->Lcap < 1 || p->Lcap > DUSTIN_MAX_LCAP) return false;
  if (p->gamma < 0 || p->k < 1 || p->sinks < 0 || p->window < 0 || p->m < 0) return false;
  if (int64_t(p->sinks) + p->window > p->k) return false;
  return true;
}

bool kv_ok(const dustin_kv& v, int Lcap) {
  if (!v.ptr || !aligned16(v.ptr)) return false;
  if (v.d != 64 && v.d != 128) return false;
  if (v.hkv < 1) return false;
  if (v.sb <= 0 || v.sh <= 0 || v.sl <= 0) return false;
  if ((v.sb % 8) || (v.sh % 8) || (v.sl % 8)) return false;
  if (v.sl < v.d) return false;
  return true;
}

bool ws_ok(const void* ws, size_t ws_bytes, size_t need) {
  return ws && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0 && ws_bytes >= need;
}

int* err_word(void* ws) { return reinterpret_cast<int*>(ws); }

// ----------------------------------------------------------- TMA encoding

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// TMA map over a cache view with box 64 columns x 128 rows and the 128-byte
// swizzle that the score kernel's ldmatrix addressing expects.  A densely
// packed cache [B][hkv][Lcap][d] is described as 2-D rows [B*hkv*Lcap][d]
// (rows of a box that run past one head's Lcap positions are past seq_len and
// masked); any other strides use a 4-D map (d, Lcap, hkv, B).  *rank is 2 or 4.
bool encode_cache_map(CUtensorMap* m, const dustin_kv& v, int Lcap, int B, int* rank,
                      int box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  const bool packed = v.sl == v.d && v.sh == int64_t(Lcap) * v.d && v.sb == int64_t(v.hkv) * v.sh &&
                      int64_t(B) * v.hkv * Lcap < (int64_t(1) << 31) - 256;
  CUresult r;
  if (packed) {
    cuuint64_t dims[2] = {cuuint64_t(v.d), cuuint64_t(B) * v.hkv * Lcap};
    cuuint64_t strides[1] = {cuuint64_t(v.sl) * 2};
    cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, v.ptr, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *rank = 2;
  } else {
    cuuint64_t dims[4] = {cuuint64_t(v.d), cuuint64_t(Lcap), cuuint64_t(v.hkv), cuuint64_t(B)};
    cuuint64_t strides[3] = {cuuint64_t(v.sl) * 2, cuuint64_t(v.sh) * 2, cuuint64_t(v.sb) * 2};
    cuuint32_t box[4] = {64, cuuint32_t(box_rows), 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v.ptr, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *rank = 4;
  }
  return r == CUDA_SUCCESS;
}

// Verify queries [B][T][hq][d] as 3-D (d, hq, B*T) with box (64, G, T): one
// load brings the G x T query rows of one (sequence, KV head) as rows t*G + h.
bool encode_query_map(CUtensorMap* m, const void* q, int d, int hq, int BT, int G, int T) {
  // the encoding depends on these arguments only: repeated calls on the same
  // buffers (one per layer and step) reuse the previous result
  struct Key {
    const void* q;
    int d, hq, BT, G, T;
  };
  constexpr int kSlots = 2 * DUSTIN_MAX_LAYERS;
  static thread_local Key keys[kSlots];
  static thread_local CUtensorMap maps[kSlots];
  static thread_local int next = 0;
  for (int i = 0; i < kSlots; ++i)
    if (keys[i].q == q && keys[i].d == d && keys[i].hq == hq && keys[i].BT == BT && keys[i].G == G &&
        keys[i].T == T) {
      *m = maps[i];
      return true;
    }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(hq), cuuint64_t(BT)};
  cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(hq) * d * 2};
  cuuint32_t box[3] = {64, cuuint32_t(G), cuuint32_t(T)};
  cuuint32_t estr[3] = {1, 1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  keys[next] = Key{q, d, hq, BT, G, T};
  maps[next] = *m;
  next = (next + 1) % kSlots;
  return true;
}

// ------------------------------------------------------------- score plan

// Logits of one group of sequences are kept under this size so that they stay
// in L2 (about 126 MB) between the stream and the normalise kernels.  96 MB
// scores the 16-sequence, 32 K-position batch in one group (92.5 MB of
// logits): its stream kernel then moves 0.80 of the measured HBM peak against
// 0.77 for two groups of 8, at the same step time; 48 MB split the
// 68-pair sweep points into uneven groups and cost them 10 us of scoring.
constexpr size_t kScoreL2Budget = size_t(96) << 20;

// Groups per normalise launch.  With two, the second group's stream kernel
// starts on the SMs the first one's stragglers leave and one normalise covers
// both; with a static split of each group's tiles the late-starting CTAs end
// late, which measured slower (214.7 vs 209.3 us per step at B=16, L=32k), so
// each group is normalised on its own.
constexpr int kGroupsPerNorm = 1;

struct ScorePlan {
  int n_slab = 0;
  int n_cache = 0;
  int cache_channel[DUSTIN_MAX_SRH];
  int cache_layer[DUSTIN_MAX_SRH];
  ScoreSlab slab[DUSTIN_MAX_SRH];
  int np_max = 0;
  int LSP = 0;           // logits row stride (floats, multiple of 32)
  int nb = 0;            // sequences per group
  int max_seg = 0;
  int n_rows = 0, n_rows0 = 0;
  ScoreLaunch launch{};
  // logits and statistics buffers: one per group of a pair (the second group
  // of a pair streams into its own buffers while the first one's complete)
  int n_buf = 1;
  size_t logits_off[2] = {0, 0}, logits_bytes = 0, stats_off[2] = {0, 0}, stats_bytes = 0, total = 0;
  // selection scratch of the fused step, after the score scratch
  SelectPlan sel{};
  size_t hist_off = 0, total_step = 0;
};

const dustin_signal* sig_of(int ch, const dustin_signal* draft, const dustin_signal* target) {
  return ch == 0 ? draft : target;
}

bool signal_ok(const dustin_signal* s) {
  return s && s->n_layers >= 1 && s->n_layers <= 4096 && s->hq >= 1 && s->nq >= 1 && s->q && s->k;
}

// Validates the SRH list and plans the score launches.  scratch_off is where
// the scratch begins in the workspace and scratch_max bounds it (0: no bound
// beyond the L2 budget).
int build_score_plan(const dustin_params* p, const dustin_signal* draft,
                     const dustin_signal* target, const dustin_srh* srh, int32_t n_srh,
                     ScorePlan* pl, size_t scratch_off = kScratch, size_t scratch_max = 0) {
  if (!params_ok(p)) return DUSTIN_EINVAL;
  if (!srh || n_srh < 1) return DUSTIN_EINVAL;
  if (n_srh > DUSTIN_MAX_SRH) return DUSTIN_ERANGE;
  std::memset(pl, 0, sizeof(*pl));
  for (int i = 0; i < n_srh; ++i) {
    const dustin_srh& e = srh[i];
    if (e.channel != 0 && e.channel != 1) return DUSTIN_EINVAL;
    const dustin_signal* s = sig_of(e.channel, draft, target);
    if (!signal_ok(s)) return DUSTIN_EINVAL;
    if (e.layer < 0 || e.layer >= s->n_layers) return DUSTIN_EINVAL;
    if (e.q_head < 0 || e.q_head >= s->hq) return DUSTIN_EINVAL;
    for (int j = 0; j < i; ++j)
      if (srh[j].channel == e.channel && srh[j].layer == e.layer && srh[j].q_head == e.q_head)
        return DUSTIN_EINVAL;   // duplicate SRH
    const dustin_kv& kv = s->k[e.layer];
    const void* q = s->q[e.layer];
    if (!kv_ok(kv, p->Lcap) || !q || !aligned16(q)) return DUSTIN_EINVAL;
    if (s->hq % kv.hkv) return DUSTIN_EINVAL;
    const int g = e.q_head / (s->hq / kv.hkv);
    int ci = -1;
    for (int c = 0; c < pl->n_cache; ++c)
      if (pl->cache_channel[c] == e.channel && pl->cache_layer[c] == e.layer) ci = c;
    if (ci < 0) {
      ci = pl->n_cache++;
      pl->cache_channel[ci] = e.channel;
      pl->cache_layer[ci] = e.layer;
    }
    int sj = -1;
    for (int t = 0; t < pl->n_slab; ++t)
      if (pl->slab[t].cache == ci && pl->slab[t].g == g) sj = t;
    if (sj < 0) {
      sj = pl->n_slab++;
      ScoreSlab& S = pl->slab[sj];
      S.channel = e.channel;
      S.cache = ci;
      S.g = g;
      S.D = kv.d;
      S.nq = s->nq;
      S.hq = s->hq;
      S.nheads = 0;
      S.npairs = 0;
      S.rows = score_rows_per_tile(kv.d);
      S.cost = 0;
      S.tiles = (p->Lcap + S.rows - 1) / S.rows;
      S.q = static_cast<const uint16_t*>(q);
    }
    ScoreSlab& S = pl->slab[sj];
    if (S.npairs + s->nq > DUSTIN_MAX_PAIRS) return DUSTIN_ERANGE;
    S.heads[S.nheads++] = e.q_head;
    S.npairs += s->nq;
  }
  for (int t = 0; t < pl->n_slab; ++t)
    pl->slab[t].cost = score_tile_cost(pl->slab[t].D, pl->slab[t].npairs);
  pl->LSP = (p->Lcap + 31) / 32 * 32;
  size_t per_b = 0;   // logits bytes of one sequence
  for (int t = 0; t < pl->n_slab; ++t) {
    pl->np_max = pl->np_max > pl->slab[t].npairs ? pl->np_max : pl->slab[t].npairs;
    per_b += size_t(pl->slab[t].npairs) * pl->LSP * 4;
  }
  // sequences per group: logits within the L2 budget (and the scratch bound)
  size_t budget = kScoreL2Budget;
  if (scratch_max) {
    const size_t avail = scratch_max > scratch_off ? scratch_max - scratch_off : 0;
    budget = avail < budget ? avail : budget;
  }
  long long nb = (long long)(budget / (per_b + 1));
  if (nb >= 1 && nb < p->B) {   // as many groups as needed, of near-equal size
    const long long groups = (p->B + nb - 1) / nb;
    nb = (p->B + groups - 1) / groups;
  }
  for (;;) {
    if (nb > p->B) nb = p->B;
    if (nb < 1) {
      if (scratch_max) return DUSTIN_ERANGE;   // a hard scratch bound: refuse
      nb = 1;                                  // one sequence at a time, past the L2 budget
    }
    // statistics slots: a CTA's share of the cost is at least the cheapest
    // tile's cost (the grid never exceeds the tile count), so a run of `tiles`
    // tiles spans at most tiles * cost_max / cost_min + 2 CTA indices
    int tmax = 0, wmin = 1 << 30, wmax = 0;
    for (int t = 0; t < pl->n_slab; ++t) {
      tmax = tmax > pl->slab[t].tiles ? tmax : pl->slab[t].tiles;
      wmin = wmin < pl->slab[t].cost ? wmin : pl->slab[t].cost;
      wmax = wmax > pl->slab[t].cost ? wmax : pl->slab[t].cost;
    }
    pl->max_seg = int((long long)tmax * wmax / wmin) + 3;
    pl->nb = int(nb);
    pl->n_buf = (kGroupsPerNorm > 1 && p->B > nb) ? 2 : 1;
    pl->logits_bytes = round256(per_b * nb);
    pl->stats_bytes = round256(size_t(pl->n_slab) * nb * pl->max_seg * pl->np_max * 2 * 4);
    pl->logits_off[0] = scratch_off;
    pl->logits_off[1] = scratch_off + pl->logits_bytes;
    pl->stats_off[0] = scratch_off + pl->n_buf * pl->logits_bytes;
    pl->stats_off[1] = pl->stats_off[0] + pl->stats_bytes;
    pl->total = pl->stats_off[0] + pl->n_buf * pl->stats_bytes;
    if (!scratch_max || pl->total <= scratch_max) break;
    --nb;
  }
  long long off = 0;
  for (int t = 0; t < pl->n_slab; ++t) {
    pl->slab[t].logit_off = off;
    off += (long long)pl->nb * pl->slab[t].npairs * pl->LSP;
  }
  // logits rows per sequence (channel 0 first)
  for (int t = 0; t < pl->n_slab; ++t) {
    pl->n_rows += pl->slab[t].npairs;
    if (pl->slab[t].channel == 0) pl->n_rows0 += pl->slab[t].npairs;
  }
  // the fused step's selection scratch (its histograms first) follows the
  // score scratch: the normalise kernel fills the histograms
  pl->sel = select_plan(p->B, p->Lcap, pl->total);
  pl->hist_off = pl->sel.hist_off;
  pl->total_step = pl->sel.end;
  pl->launch.NT = (pl->np_max + 7) / 8;
  pl->launch.smem = score_stream_smem();
  pl->launch.norm_smem = score_norm_smem(pl->n_rows);
  return DUSTIN_OK;
}

// hist: the selection histograms to build (fused step), or nullptr.
int launch_score(const dustin_params* p, const dustin_signal* draft, const dustin_signal* target,
                 const ScorePlan& pl, const int32_t* seq_len, float* importance, void* ws,
                 cudaStream_t stream, cudaEvent_t after_first_stream = nullptr,
                 int* hist = nullptr) {
  static thread_local ScoreArgs a;   // large (tensor maps): keep it off the stack
  std::memset(&a, 0, sizeof(a));
  int rank[DUSTIN_MAX_SRH];
  for (int c = 0; c < pl.n_cache; ++c) {
    const dustin_signal* s = sig_of(pl.cache_channel[c], draft, target);
    if (!encode_cache_map(&a.map[c], s->k[pl.cache_layer[c]], p->Lcap, p->B, &rank[c]))
      return DUSTIN_ECUDA;
  }
  for (int t = 0; t < pl.n_slab; ++t) {
    a.slab[t] = pl.slab[t];
    const dustin_signal* s = sig_of(pl.slab[t].channel, draft, target);
    a.slab[t].row2d = rank[pl.slab[t].cache] == 2 ? s->k[pl.cache_layer[pl.slab[t].cache]].hkv : 0;
  }
  a.B = p->B;
  a.Lcap = p->Lcap;
  a.LSP = pl.LSP;
  a.n_slab = pl.n_slab;
  a.np_max = pl.np_max;
  a.max_seg = pl.max_seg;
  a.seq_len = seq_len;
  a.err = err_word(ws);
  a.importance = importance;
  a.hist = hist;
  a.sinks = p->sinks;
  a.window = p->window;
  a.n_rows = pl.n_rows;
  a.n_rows0 = pl.n_rows0;
  const int sms = num_sms() > 0 ? num_sms() : 148;
  long long wmax = 1;   // every CTA's share must reach the largest tile cost,
  for (int t = 0; t < pl.n_slab; ++t)   // so that each CTA owns a tile
    if (pl.slab[t].cost > wmax) wmax = pl.slab[t].cost;
  const int nchunks = (pl.LSP + 255) / 256;
  // Groups of nb sequences go kGroupsPerNorm at a time: their stream kernels
  // (each group but the first of a batch into its own buffers, started
  // without waiting so that it fills the SMs the previous group's stragglers
  // leave), then one normalise over them.
  for (int pb = 0; pb < p->B; pb += kGroupsPerNorm * pl.nb) {
    a.n_groups = 0;
    for (int gr = 0; gr < kGroupsPerNorm; ++gr) {
      const int b0 = pb + gr * pl.nb;
      if (b0 >= p->B) break;
      a.b0 = b0;
      a.nb = p->B - b0 < pl.nb ? p->B - b0 : pl.nb;
      a.logits = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.logits_off[gr]);
      a.stats = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.stats_off[gr]);
      a.wait_at_end = gr;
      long long acc = 0, cost = 0;
      for (int t = 0; t < pl.n_slab; ++t) {
        a.slab_start[t] = acc;
        a.cost_start[t] = cost;
        acc += (long long)a.nb * pl.slab[t].tiles;
        cost += (long long)a.nb * pl.slab[t].tiles * pl.slab[t].cost;
      }
      a.slab_start[pl.n_slab] = acc;
      a.cost_start[pl.n_slab] = cost;
      a.total = acc;
      a.total_cost = cost;
      long long grid = sms < kScoreGridMax ? sms : kScoreGridMax;
      if (grid > a.total_cost / wmax) grid = a.total_cost / wmax;
      if (grid < 1) grid = 1;
      a.grid = int(grid);
      // this group as the normalise kernel sees it
      NormGroup& g = a.ng[gr];
      g.b0 = a.b0;
      g.nb = a.nb;
      g.grid = a.grid;
      g.total_cost = a.total_cost;
      g.logits = a.logits;
      g.stats = a.stats;
      int n_info = 0, row = 0;   // the slabs in logits-row order: channel 0 first
      for (int ch = 0; ch < 2; ++ch)
        for (int t = 0; t < pl.n_slab; ++t) {
          if (pl.slab[t].channel != ch) continue;
          SlabInfo& I = a.info[gr][n_info++];
          I.logit_off = pl.slab[t].logit_off;
          I.first_tile = a.slab_start[t];
          I.cost_start = a.cost_start[t];
          I.npairs = pl.slab[t].npairs;
          I.tiles = pl.slab[t].tiles;
          I.cost = pl.slab[t].cost;
          I.row0 = row;
          I.slab = t;
          I.pad = 0;
          row += pl.slab[t].npairs;
        }
      a.n_groups = gr + 1;
      if (score_stream_launch(a, pl.launch, stream) != cudaSuccess) return DUSTIN_ECUDA;
      if (pb == 0 && gr == 0 && after_first_stream &&
          cudaEventRecord(after_first_stream, stream) != cudaSuccess)
        return DUSTIN_ECUDA;
    }
    // normalise both: every CTA resident at once, spread over the sequences
    int nseq = 0;
    for (int gr = 0; gr < a.n_groups; ++gr) nseq += a.ng[gr].nb;
    int cps = int((long long)sms * score_norm_ctas_per_sm(pl.n_rows) / nseq);
    if (cps < 1) cps = 1;
    if (cps > nchunks) cps = nchunks;
    for (int gr = 0; gr < a.n_groups; ++gr) a.ng[gr].cps = cps;
    if (score_norm_launch(a, pl.launch, stream) != cudaSuccess) return DUSTIN_ECUDA;
  }
  return DUSTIN_OK;
}

// ----------------------------------------------------------- verify setup

int check_verify_layer(const dustin_params* p, int32_t hq, const void* q, const dustin_kv& k,
                       const dustin_kv& v, const void* kb, const void* vb, const float* o) {
  if (!q || !kb || !vb || !o) return DUSTIN_EINVAL;
  if (!aligned16(q) || !aligned16(kb) || !aligned16(vb) || !aligned16(o)) return DUSTIN_EINVAL;
  if (!kv_ok(k, p->Lcap) || !kv_ok(v, p->Lcap)) return DUSTIN_EINVAL;
  if (k.hkv != v.hkv || k.d != v.d) return DUSTIN_EINVAL;
  if (hq < 1 || hq % k.hkv) return DUSTIN_EINVAL;
  const int64_t nq = int64_t(p->gamma + 1) * (hq / k.hkv);
  if (nq > DUSTIN_MAX_QROWS || p->gamma + 1 > DUSTIN_MAX_BLOCK) return DUSTIN_ERANGE;
  return DUSTIN_OK;
}

void fill_layer(VerifyLayerDev& L, const void* q, const dustin_kv& k, const dustin_kv& v,
                const void* kb, const void* vb, float* o) {
  L.q = static_cast<const uint16_t*>(q);
  L.k = static_cast<const uint16_t*>(k.ptr);
  L.v = static_cast<const uint16_t*>(v.ptr);
  L.kb = static_cast<const uint16_t*>(kb);
  L.vb = static_cast<const uint16_t*>(vb);
  L.o = o;
  L.ksb = k.sb; L.ksh = k.sh; L.ksl = k.sl;
  L.vsb = v.sb; L.vsh = v.sh; L.vsl = v.sl;
}

struct VerifyShape {
  int hq = 0, hkv = 0, d = 0, n_layers = 0;
};

VerifyLaunch plan_verify(const dustin_params* p, const VerifyShape& v, int dense) {
  const int NQ = (p->gamma + 1) * (v.hq / v.hkv);
  return verify_plan(v.d, NQ, dense ? p->Lcap : p->k, p->B, v.hkv, v.n_layers, dense, num_sms());
}

// Bytes of workspace the verification of this shape needs (0 if invalid).
size_t verify_ws_bytes(const dustin_params* p, const VerifyShape& v, int dense) {
  if (v.n_layers <= 0) return kScratch;
  const VerifyLaunch pl = plan_verify(p, v, dense);
  if (pl.units > kVerifyUnitsMax) return 0;
  return kScratch + round256(verify_scratch_bytes(pl));
}

int run_verify(const dustin_params* p, int32_t hq, int hkv, int D, int n_layers,
               const VerifyLayerDev* layers, const int32_t* ivf, const int32_t* seq_len, int dense,
               void* ws, size_t ws_bytes, cudaStream_t stream) {
  VerifyShape vs;
  vs.hq = hq;
  vs.hkv = hkv;
  vs.d = D;
  vs.n_layers = n_layers;
  const VerifyLaunch pl = plan_verify(p, vs, dense);
  if (pl.units > kVerifyUnitsMax) return DUSTIN_ERANGE;
  if (!ws_ok(ws, ws_bytes, kScratch + verify_scratch_bytes(pl))) return DUSTIN_EWORKSPACE;
  static thread_local VerifyArgs a;
  std::memset(&a, 0, sizeof(a));
  a.B = p->B;
  a.Lcap = p->Lcap;
  a.T = p->gamma + 1;
  a.hq = hq;
  a.hkv = hkv;
  a.G = hq / hkv;
  a.NQ = a.T * a.G;
  a.k = p->k;
  a.dense = dense;
  a.n_layers = n_layers;
  a.ctx_tiles = pl.ctx_tiles;
  a.tiles_u = pl.tiles_u;
  a.total = pl.total;
  a.max_seg = pl.max_seg;
  a.slot_floats = pl.slot_floats;
  a.scale_log2 = float(1.4426950408889634 / std::sqrt(double(D)));
  a.lay = pl.lay;
  a.ivf = ivf;
  a.seq_len = seq_len;
  a.err = err_word(ws);
  a.partial = reinterpret_cast<float*>(static_cast<char*>(ws) + kScratch);
  for (int l = 0; l < n_layers; ++l) {
    const VerifyLayerDev& L = layers[l];
    a.layer[l] = L;
    if (!encode_query_map(&a.qmap[l], L.q, D, hq, p->B * a.T, a.G, a.T)) return DUSTIN_ECUDA;
  }
  // dense: contiguous context tiles by TMA boxes when every cache can be
  // described by a tensor map (else the row gathers serve every tile)
  a.tma = dense ? 1 : 0;
  for (int l = 0; l < n_layers && a.tma; ++l) {
    const VerifyLayerDev& L = layers[l];
    const dustin_kv kv{const_cast<uint16_t*>(L.k), hkv, D, L.ksb, L.ksh, L.ksl};
    const dustin_kv vv{const_cast<uint16_t*>(L.v), hkv, D, L.vsb, L.vsh, L.vsl};
    int rk = 0, rv = 0;   // boxes of one 64-key tile
    if (!encode_cache_map(&a.kmap[l], kv, p->Lcap, p->B, &rk, DUSTIN_MAX_BLOCK) ||
        !encode_cache_map(&a.vmap[l], vv, p->Lcap, p->B, &rv, DUSTIN_MAX_BLOCK) || rk != rv)
      a.tma = 0;
    a.kvrank[l] = rk;
  }
  if (verify_launch(a, pl, stream) != cudaSuccess) return DUSTIN_ECUDA;
  return DUSTIN_OK;
}

}  // namespace

extern "C" {

const char* dustin_version(void) { return "dustin-gb300 0.1 (sm_103a)"; }

size_t dustin_workspace_bytes(const dustin_params* p, const dustin_signal* draft,
                              const dustin_signal* target, const dustin_srh* srh, int32_t n_srh,
                              int32_t hq, int32_t hkv, int32_t d, int32_t n_layers) {
  if (!params_ok(p)) return 0;
  size_t need = select_plan(p->B, p->Lcap, kScratch).end;   // dustin_select
  if (n_srh != 0) {
    static thread_local ScorePlan pl;
    if (build_score_plan(p, draft, target, srh, n_srh, &pl) != DUSTIN_OK) return 0;
    need = pl.total_step > need ? pl.total_step : need;
  }
  if (n_layers != 0) {
    if (n_layers < 0 || n_layers > DUSTIN_MAX_LAYERS || hkv < 1 || hq < 1 || hq % hkv ||
        (d != 64 && d != 128) || int64_t(p->gamma + 1) * (hq / hkv) > DUSTIN_MAX_QROWS ||
        p->gamma + 1 > DUSTIN_MAX_BLOCK)
      return 0;
    VerifyShape vs;
    vs.hq = hq;
    vs.hkv = hkv;
    vs.d = d;
    vs.n_layers = n_layers;
    for (int dense = 0; dense < 2; ++dense) {
      const size_t v = verify_ws_bytes(p, vs, dense);
      if (v == 0) return 0;
      need = v > need ? v : need;
    }
  }
  return need;
}

int dustin_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!ws_ok(ws, ws_bytes, kScratch)) return DUSTIN_EWORKSPACE;
  return cudaMemsetAsync(ws, 0, kScratch, stream) == cudaSuccess ? DUSTIN_OK : DUSTIN_ECUDA;
}

int dustin_check(void* ws, cudaStream_t stream, int32_t* flags) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DUSTIN_EWORKSPACE;
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return DUSTIN_ECUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DUSTIN_ECUDA;
  if (flags) *flags = h;
  if (h != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof(h), stream) != cudaSuccess) return DUSTIN_ECUDA;
    return DUSTIN_EDEVICE;
  }
  return DUSTIN_OK;
}

int dustin_score(const dustin_params* p, const dustin_signal* draft, const dustin_signal* target,
                 const dustin_srh* srh, int32_t n_srh, const int32_t* seq_len, float* importance,
                 void* ws, size_t ws_bytes, cudaStream_t stream) {
  static thread_local ScorePlan pl;
  const int st = build_score_plan(p, draft, target, srh, n_srh, &pl);
  if (st != DUSTIN_OK) return st;
  if (!seq_len || !importance || !aligned16(importance)) return DUSTIN_EINVAL;
  if (!ws_ok(ws, ws_bytes, pl.total)) return DUSTIN_EWORKSPACE;
  return launch_score(p, draft, target, pl, seq_len, importance, ws, stream);
}

}  // extern "C"

namespace {

// sel: the selection scratch; fused: its histograms were built by the score
// kernels of this call (otherwise select_launch counts them first).
int run_select(const dustin_params* p, const float* importance, const int32_t* seq_len,
               int32_t* i_verify, const SelectPlan& sel, bool fused, void* ws, size_t ws_bytes,
               cudaStream_t stream) {
  if (!params_ok(p)) return DUSTIN_EINVAL;
  if (!importance || !seq_len || !i_verify) return DUSTIN_EINVAL;
  if (!ws_ok(ws, ws_bytes, sel.end)) return DUSTIN_EWORKSPACE;
  char* w = static_cast<char*>(ws);
  SelectArgs a{};
  a.hist = reinterpret_cast<int*>(w + sel.hist_off);
  a.bits = reinterpret_cast<uint32_t*>(w + sel.bits_off);
  a.bits_words = sel.bits_words;
  a.B = p->B;
  a.Lcap = p->Lcap;
  a.k = p->k;
  a.sinks = p->sinks;
  a.window = p->window;
  a.m = p->m;
  a.imp = importance;
  a.seq_len = seq_len;
  a.out = i_verify;
  a.err = err_word(ws);
  return select_launch(a, !fused, stream) == cudaSuccess ? DUSTIN_OK : DUSTIN_ECUDA;
}

}  // namespace

extern "C" {

int dustin_select(const dustin_params* p, const float* importance, const int32_t* seq_len,
                  int32_t* i_verify, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!params_ok(p)) return DUSTIN_EINVAL;
  return run_select(p, importance, seq_len, i_verify, select_plan(p->B, p->Lcap, kScratch), false, ws,
                    ws_bytes, stream);
}

int dustin_verify_attn(const dustin_params* p, int32_t hq, const void* q, dustin_kv k,
                       dustin_kv v, const void* kb, const void* vb, const int32_t* i_verify,
                       const int32_t* seq_len, float* o, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
  if (!params_ok(p)) return DUSTIN_EINVAL;
  const int st = check_verify_layer(p, hq, q, k, v, kb, vb, o);
  if (st != DUSTIN_OK) return st;
  if (!i_verify || !seq_len) return DUSTIN_EINVAL;
  if (!ws_ok(ws, ws_bytes, kScratch)) return DUSTIN_EWORKSPACE;
  VerifyLayerDev L;
  fill_layer(L, q, k, v, kb, vb, o);
  return run_verify(p, hq, k.hkv, k.d, 1, &L, i_verify, seq_len, 0, ws, ws_bytes, stream);
}

int dense_verify_attn(const dustin_params* p, int32_t hq, const void* q, dustin_kv k, dustin_kv v,
                      const void* kb, const void* vb, const int32_t* seq_len, float* o, void* ws,
                      size_t ws_bytes, cudaStream_t stream) {
  if (!params_ok(p)) return DUSTIN_EINVAL;
  const int st = check_verify_layer(p, hq, q, k, v, kb, vb, o);
  if (st != DUSTIN_OK) return st;
  if (!seq_len) return DUSTIN_EINVAL;
  if (!ws_ok(ws, ws_bytes, kScratch)) return DUSTIN_EWORKSPACE;
  VerifyLayerDev L;
  fill_layer(L, q, k, v, kb, vb, o);
  return run_verify(p, hq, k.hkv, k.d, 1, &L, nullptr, seq_len, 1, ws, ws_bytes, stream);
}

int dustin_kv_append(const dustin_params* p, int32_t n_layers, const dustin_kv* k,
                     const dustin_kv* v, const void* const* kb, const void* const* vb,
                     const int32_t* n_accept, int32_t* seq_len, void* ws, size_t ws_bytes,
                     cudaStream_t stream) {
  if (!params_ok(p)) return DUSTIN_EINVAL;
  if (n_layers < 1) return DUSTIN_EINVAL;
  if (n_layers > DUSTIN_MAX_LAYERS) return DUSTIN_ERANGE;
  if (!k || !v || !kb || !vb || !n_accept || !seq_len) return DUSTIN_EINVAL;
  if (!ws_ok(ws, ws_bytes, kScratch)) return DUSTIN_EWORKSPACE;
  AppendArgs a{};
  a.B = p->B;
  a.Lcap = p->Lcap;
  a.T = p->gamma + 1;
  a.hkv = k[0].hkv;
  a.D = k[0].d;
  a.n_layers = n_layers;
  a.n_accept = n_accept;
  a.seq_len = seq_len;
  a.err = err_word(ws);
  for (int l = 0; l < n_layers; ++l) {
    if (!kv_ok(k[l], p->Lcap) || !kv_ok(v[l], p->Lcap)) return DUSTIN_EINVAL;
    if (k[l].hkv != a.hkv || v[l].hkv != a.hkv || k[l].d != a.D || v[l].d != a.D)
      return DUSTIN_EINVAL;
    if (!kb[l] || !vb[l] || !aligned16(kb[l]) || !aligned16(vb[l])) return DUSTIN_EINVAL;
    AppendLayerDev& L = a.layer[l];
    L.k = static_cast<uint16_t*>(k[l].ptr);
    L.v = static_cast<uint16_t*>(v[l].ptr);
    L.kb = static_cast<const uint16_t*>(kb[l]);
    L.vb = static_cast<const uint16_t*>(vb[l]);
    L.ksb = k[l].sb; L.ksh = k[l].sh; L.ksl = k[l].sl;
    L.vsb = v[l].sb; L.vsh = v[l].sh; L.vsl = v[l].sl;
  }
  return append_launch(a, stream) == cudaSuccess ? DUSTIN_OK : DUSTIN_ECUDA;
}

int dustin_compact_kv(const dustin_params* p, int32_t n_layers, const dustin_kv* k,
                      const dustin_kv* v, const int32_t* i_verify, const int32_t* seq_len,
                      const dustin_kv* kc, const dustin_kv* vc, int32_t* seq_len_c, void* ws,
                      size_t ws_bytes, cudaStream_t stream) {
  if (!params_ok(p)) return DUSTIN_EINVAL;
  if (n_layers < 1) return DUSTIN_EINVAL;
  if (n_layers > DUSTIN_MAX_LAYERS) return DUSTIN_ERANGE;
  if (!k || !v || !kc || !vc || !i_verify || !seq_len || !seq_len_c) return DUSTIN_EINVAL;
  if (seq_len_c == seq_len) return DUSTIN_EINVAL;
  if (!ws_ok(ws, ws_bytes, kScratch)) return DUSTIN_EWORKSPACE;
  CompactArgs a{};
  a.B = p->B;
  a.Lcap = p->Lcap;
  a.k = p->k;
  a.hkv = k[0].hkv;
  a.D = k[0].d;
  a.n_layers = n_layers;
  a.ivf = i_verify;
  a.seq_len = seq_len;
  a.seq_len_c = seq_len_c;
  a.err = err_word(ws);
  for (int l = 0; l < n_layers; ++l) {
    if (!kv_ok(k[l], p->Lcap) || !kv_ok(v[l], p->Lcap)) return DUSTIN_EINVAL;
    if (!kv_ok(kc[l], p->k) || !kv_ok(vc[l], p->k)) return DUSTIN_EINVAL;
    for (const dustin_kv* t : {&k[l], &v[l], &kc[l], &vc[l]})
      if (t->hkv != a.hkv || t->d != a.D) return DUSTIN_EINVAL;
    CompactLayerDev& L = a.layer[l];
    L.k = static_cast<const uint16_t*>(k[l].ptr);
    L.v = static_cast<const uint16_t*>(v[l].ptr);
    L.kc = static_cast<uint16_t*>(const_cast<void*>(kc[l].ptr));
    L.vc = static_cast<uint16_t*>(const_cast<void*>(vc[l].ptr));
    L.ksb = k[l].sb; L.ksh = k[l].sh; L.ksl = k[l].sl;
    L.vsb = v[l].sb; L.vsh = v[l].sh; L.vsl = v[l].sl;
    L.kcsb = kc[l].sb; L.kcsh = kc[l].sh; L.kcsl = kc[l].sl;
    L.vcsb = vc[l].sb; L.vcsh = vc[l].sh; L.vcsl = vc[l].sl;
  }
  return compact_launch(a, stream) == cudaSuccess ? DUSTIN_OK : DUSTIN_ECUDA;
}

int dustin_step_launches(const dustin_step* s, int32_t* n_launches, int32_t* group_size) {
  if (!s || !n_launches || !group_size) return DUSTIN_EINVAL;
  static thread_local ScorePlan pl;
  const int st = build_score_plan(&s->p, s->draft, s->target, s->srh, s->n_srh, &pl);
  if (st != DUSTIN_OK) return st;
  const int groups = (s->p.B + pl.nb - 1) / pl.nb;
  // a stream kernel per group, a normalise per kGroupsPerNorm groups, select,
  // verify + merge
  *n_launches = groups + (groups + kGroupsPerNorm - 1) / kGroupsPerNorm + 3;
  *group_size = pl.nb;
  return DUSTIN_OK;
}

int dustin_verify_split(const dustin_params* p, int32_t hq, int32_t hkv, int32_t d,
                        int32_t n_layers, int32_t dense, int32_t* grid, int32_t* tiles_per_unit) {
  if (!params_ok(p) || !grid || !tiles_per_unit) return DUSTIN_EINVAL;
  if (n_layers < 1 || n_layers > DUSTIN_MAX_LAYERS || hkv < 1 || hq < 1 || hq % hkv ||
      (d != 64 && d != 128))
    return DUSTIN_EINVAL;
  if (int64_t(p->gamma + 1) * (hq / hkv) > DUSTIN_MAX_QROWS || p->gamma + 1 > DUSTIN_MAX_BLOCK)
    return DUSTIN_ERANGE;
  VerifyShape vs;
  vs.hq = hq;
  vs.hkv = hkv;
  vs.d = d;
  vs.n_layers = n_layers;
  const VerifyLaunch pl = plan_verify(p, vs, dense ? 1 : 0);
  if (pl.units > kVerifyUnitsMax) return DUSTIN_ERANGE;
  *grid = pl.grid;
  *tiles_per_unit = pl.tiles_u;
  return DUSTIN_OK;
}

int dustin_verify_step(const dustin_step* s, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!s) return DUSTIN_EINVAL;
  const dustin_params* p = &s->p;
  static thread_local ScorePlan pl;
  int st = build_score_plan(p, s->draft, s->target, s->srh, s->n_srh, &pl);
  if (st != DUSTIN_OK) return st;
  if (!s->seq_len || !s->importance || !aligned16(s->importance) || !s->i_verify)
    return DUSTIN_EINVAL;
  if (s->n_layers < 1 || !s->layers) return DUSTIN_EINVAL;
  if (s->n_layers > DUSTIN_MAX_LAYERS) return DUSTIN_ERANGE;
  VerifyLayerDev layers[DUSTIN_MAX_LAYERS];
  const int hkv = s->layers[0].k.hkv, D = s->layers[0].k.d;
  for (int l = 0; l < s->n_layers; ++l) {
    const dustin_verify_layer& V = s->layers[l];
    st = check_verify_layer(p, s->hq, V.q, V.k, V.v, V.kb, V.vb, V.o);
    if (st != DUSTIN_OK) return st;
    if (V.k.hkv != hkv || V.k.d != D) return DUSTIN_EINVAL;
    fill_layer(layers[l], V.q, V.k, V.v, V.kb, V.vb, V.o);
  }
  VerifyShape vs;
  vs.hq = s->hq;
  vs.hkv = hkv;
  vs.d = D;
  vs.n_layers = s->n_layers;
  const size_t vneed = verify_ws_bytes(p, vs, 0);
  if (vneed == 0) return DUSTIN_ERANGE;
  if (!ws_ok(ws, ws_bytes, pl.total_step > vneed ? pl.total_step : vneed)) return DUSTIN_EWORKSPACE;
  int* hist = reinterpret_cast<int*>(static_cast<char*>(ws) + pl.hist_off);
  cudaEvent_t* ev = s->stage_events;
  if (ev && cudaEventRecord(ev[0], stream) != cudaSuccess) return DUSTIN_ECUDA;
  st = launch_score(p, s->draft, s->target, pl, s->seq_len, s->importance, ws, stream,
                    ev ? ev[1] : nullptr, hist);
  if (st != DUSTIN_OK) return st;
  if (ev && cudaEventRecord(ev[2], stream) != cudaSuccess) return DUSTIN_ECUDA;
  st = run_select(p, s->importance, s->seq_len, s->i_verify, pl.sel, true, ws, ws_bytes, stream);
  if (st != DUSTIN_OK) return st;
  if (ev && cudaEventRecord(ev[3], stream) != cudaSuccess) return DUSTIN_ECUDA;
  st = run_verify(p, s->hq, hkv, D, s->n_layers, layers, s->i_verify, s->seq_len, 0, ws, ws_bytes,
                  stream);
  if (st != DUSTIN_OK) return st;
  if (ev && cudaEventRecord(ev[4], stream) != cudaSuccess) return DUSTIN_ECUDA;
  return DUSTIN_OK;
}

int dustin_wait_selftest(int64_t limit_ns, int64_t* waited_ns, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000ll) return DUSTIN_EINVAL;
  if (!waited_ns || (reinterpret_cast<uintptr_t>(waited_ns) & 7u)) return DUSTIN_EINVAL;
  if (!ws_ok(ws, ws_bytes, kHeader)) return DUSTIN_EWORKSPACE;
  return wait_selftest_launch(err_word(ws), reinterpret_cast<long long*>(waited_ns),
                              static_cast<unsigned long long>(limit_ns), stream) == cudaSuccess
             ? DUSTIN_OK
             : DUSTIN_ECUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Scoring without a caller workspace (for callers that cannot allocate).
// The scratch is this file-scope device array; host code must not use its
// name as a device address, so the address is looked up per device.
// ---------------------------------------------------------------------------

static __device__ __align__(256) unsigned char g_noalloc_scratch[DUSTIN_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device (looked up once
// per device, with that device current).  The first lookup on a device also
// clears the array's error word, on the caller's stream, so the word starts
// from zero whatever the loader left in the array.
int noalloc_scratch(void** out, cudaStream_t stream) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DUSTIN_ECUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DUSTIN_ECUDA;
    if (cudaMemsetAsync(p, 0, kHeader, stream) != cudaSuccess) return DUSTIN_ECUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return DUSTIN_OK;
}

}  // namespace

extern "C" int dustin_score_noalloc(const dustin_params* p, const dustin_signal* draft,
                                    const dustin_signal* target, const dustin_srh* srh,
                                    int32_t n_srh, const int32_t* seq_len, float* importance,
                                    cudaStream_t stream) {
  static thread_local ScorePlan pl;
  const int st = build_score_plan(p, draft, target, srh, n_srh, &pl, kHeader,
                                  DUSTIN_NOALLOC_SCRATCH_BYTES);
  if (st != DUSTIN_OK) return st;
  if (!seq_len || !importance || !aligned16(importance)) return DUSTIN_EINVAL;
  if (pl.total > DUSTIN_NOALLOC_SCRATCH_BYTES) return DUSTIN_ERANGE;
  void* ws = nullptr;
  const int s2 = noalloc_scratch(&ws, stream);
  if (s2 != DUSTIN_OK) return s2;
  return launch_score(p, draft, target, pl, seq_len, importance, ws, stream);
}

extern "C" int dustin_score_noalloc_check(cudaStream_t stream, int32_t* flags) {
  void* ws = nullptr;
  const int st = noalloc_scratch(&ws, stream);
  if (st != DUSTIN_OK) return st;
  return dustin_check(ws, stream, flags);
}
