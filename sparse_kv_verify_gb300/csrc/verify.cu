// Sparse and dense verification attention ("Technical Summary: Dustin",
// section 3 "Verification Workflow", steps 3-4; the dense comparator follows
// the "Problem Statement": standard verification loads the whole cache).
//
// Work: for every (layer, sequence b, KV head g) "unit", the (gamma+1) x G
// query rows that share KV head g attend to the unit's key rows (sparse: the
// entries of I_verify; dense: positions 0..seq_len-1) plus the gamma+1
// draft-block rows under the causal mask u <= t.
//
// Schedule (stream-K): each unit is cut into 64-key tiles followed by one
// block tile; all units' tiles form one sequence that is split evenly over the
// persistent CTAs (two per SM when the query rows fit 64-row MMAs and two
// CTAs' shared memory fits an SM, else one), so every CTA moves the same
// number of bytes whatever B, Hkv and k are.  Two CTAs per SM gather faster
// than one: each drains its ring in order, and two rings cover each other's
// late rows.
//
// Roles inside a CTA (warp specialised, handing over through mbarriers):
//   warps 4-11       loaders: warp w copies keys [8 (w-4), 8 (w-4) + 8) of
//   (loaders)        every tile, K and V rows, with 16-byte cp.async straight
//                    into the 128-byte-swizzled K-major layout the MMA reads
//                    (rows the tile does not use are zero-filled) through a
//                    ring of five 32 KB stages (eight 16 KB ones for d = 64;
//                    three and six with two CTAs per SM);
//                    each copy's completion arrives on the stage's barrier
//                    (cp.async.mbarrier.arrive).  A dense tile that lies wholly
//                    inside the cache comes instead as tiled TMA loads (a K
//                    and a V box of 64 rows x 64 columns per 64-column panel)
//                    issued by one loader thread.  A
//                    segment's query rows come with one tiled TMA load into one
//                    of two query buffers (one with two CTAs per SM);
//   warp 12 (S)      one thread issues S = Q K^T of each tile into one of two S
//                    buffers in tensor memory as soon as its rows have landed
//                    (after a proxy fence, since cp.async rows were written
//                    through the generic proxy);
//   warp 13 (P V)    one thread issues O += P V of each tile with P read from
//                    tensor memory, then frees the tile's stage; splitting the
//                    two MMA streams over two warps keeps one issuing thread
//                    from bounding a tile;
//   warps 0-3        one thread per query row (tensor-memory lane; warps with
//                    no query row sit the loop out): online softmax of its S
//                    row in the log2 domain, with the reference max moved only
//                    when a tile passes it by more than 2^8 (so O is rarely
//                    rescaled), P rounded to bf16 and stored back to tensor
//                    memory once the P V MMA two tiles back has read that P
//                    buffer (with two CTAs per SM, P overwrites the S buffer it
//                    came from, and the S thread waits for that P V instead);
//                    then the epilogue.
//
// Merge: a segment that covers a whole unit writes O directly; otherwise it
// writes (row max, row sum, unnormalised O) to the workspace, and a second,
// small kernel launched right behind this one merges each split unit's
// segments with a log-sum-exp combine (one thread per output float4).
#include "common.cuh"
#include "kernels.h"

namespace dustin {

namespace {

constexpr int TK = 64;           // keys per tile (and the largest draft block)
constexpr int kSoftmaxWarps = 4;    // one thread per tensor-memory lane
constexpr int kLoaders = 8;         // loader warps, kKpw keys of every tile each
constexpr int kKpw = TK / kLoaders;  // keys per loader warp and tile
constexpr int kLoaderWarp0 = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + kLoaders;
constexpr int kPvWarp = kMmaWarp + 1;   // issues the P V MMAs (kMmaWarp issues S = Q K^T)
constexpr int NTH = 32 * (kPvWarp + 1);
constexpr int kSCol = 0;         // S buffers: columns [0, 64) and [64, 128)
constexpr int kPCol = 128;       // P buffers (bf16 pairs): [128, 160) and [160, 192)
static_assert(TK == DUSTIN_MAX_BLOCK, "the draft block must fit one tile");

// Tensor-memory columns per CTA.  With one CTA per SM the P buffers sit at
// kPCol and O after them; with two CTAs per SM (256 columns each) P is stored
// over the S buffer it was computed from, and O follows the S buffers.
template <int D, int CPS>
struct TmemCfg {
  static constexpr int cols = CPS == 2 ? 256 : (D == 128 ? 512 : 256);
  static constexpr int o_col = CPS == 2 ? 128 : (D == 128 ? 256 : 192);
  static constexpr int p_col = CPS == 2 ? kSCol : kPCol;     // P buffer 0
  static constexpr int p_stride = CPS == 2 ? TK : TK / 2;    // columns from P buffer 0 to 1
};

// ---- tcgen05 ---------------------------------------------------------------

// Shared-memory operand descriptor: start, leading and stride byte offsets
// (each >> 4), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((addr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of a bf16 x bf16 -> fp32 MMA of M x N; A K-major, B
// K-major (b_mn = 0) or MN-major (b_mn = 1).
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(b_mn) << 16) | (uint32_t(N >> 3) << 17) |
         (uint32_t(M >> 4) << 24);
}

// D (tensor memory) (+)= A (shared memory) * B (shared memory)
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          int acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// D (tensor memory) (+)= A (tensor memory: one row per lane, two bf16 per
// column) * B (shared memory)
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, int acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive 32-bit columns of this thread's lane (the load and its wait
// in one statement, so that no register is read before it has landed).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// 16-lane shapes (M = 64 accumulators: rows 16 q .. 16 q + 15 in lanes 32 q ..
// 32 q + 15).  16x256b: thread t holds lanes base + t / 4 and base + 8 + t / 4,
// columns 2 (t % 4) and 2 (t % 4) + 1 of each 8-column chunk (registers 4 c ..
// 4 c + 3 for chunk c: lane t / 4 both columns, then lane 8 + t / 4).
// 16x128b: column t % 4 of each 4-column chunk, same two lanes (registers 2 c,
// 2 c + 1).
__device__ __forceinline__ void tc_ld16x256_x8(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tc_ld16x256_x4(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tc_st16x256_x4(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tc_st16x128_x8(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// ---- TMA -------------------------------------------------------------------

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// 2-D and 4-D tiled TMA loads to a shared-memory address, with an L2 policy.
__device__ __forceinline__ void tma_load_2d_u32(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_u32(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                int c2, int c3, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
// Arrive on bar once every cp.async this thread issued so far has completed
// (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Byte offset of 16-byte chunk c of row r in a [rows][64 bf16] panel with the
// 128-byte swizzle (chunk ^= row % 8; 8-row groups 1024 bytes apart).
__device__ __forceinline__ uint32_t swz(int r, int c) { return uint32_t(r) * 128u + (uint32_t(c ^ (r & 7)) << 4); }

// Bounded wait that ignores the abort flag (drains copies in flight before
// the CTA exits); giving up sets DUSTIN_DEV_TIMEOUT.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, int* err) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > kWaitLimitNs) {
      flag_error(err, DUSTIN_DEV_TIMEOUT);
      return;
    }
}


// Shared-memory layout (bytes from the 1024-aligned base), fixed per launch
// by the head dimension D and the query rows NQ:
//   query buffers [NP panels][q_rows rows][128 B] (q_rows = NQ rounded up
//   to 8; with two buffers the next segment's rows load while this one runs,
//   with one (two CTAs per SM) they wait for its last MMAs), then the K/V
//   stages [K panels | V panels] of 64 keys, then the valid-key masks, the
//   mbarriers and two words (tensor-memory base, abort).
// Once any wait gives up (DUSTIN_DEV_TIMEOUT) every role stops issuing copies
// and MMAs; before the CTA exits the loaders still wait for their copies in
// flight and the MMA thread for its MMAs, so tensor memory is freed idle.
// The S MMA reads 128 query rows per panel; the rows past q_rows fall on the
// next buffer or the ring (whatever they hold only reaches S and O rows that
// are never used: the softmax treats rows >= NQ as empty).
template <int CPS>
struct QBufsOf {
  static constexpr int n = CPS == 2 ? 1 : 2;
};
constexpr uint32_t kVerifySmem = 227 * 1024;
constexpr uint32_t kSmemPerSm = 228 * 1024;   // shared memory of an SM (1 KB reserved per CTA)

// K/V stages per head dimension and CTAs per SM (compile-time: the stage and
// phase of tile gi are gi % n and gi / n on the hot paths).  More than five
// 32 KB stages measured no faster at d = 128 with one CTA per SM (the MMA
// issue rate bounds a tile, not the bytes in flight) and slower for
// contiguous rows; two CTAs per SM hold three (d = 128) or six (d = 64) each.
template <int D, int CPS>
struct StagesOf {
  static constexpr int n = CPS == 2 ? (D == 128 ? 3 : 6) : (D == 128 ? 5 : 8);
};

inline VLay make_lay(int D, int NQ, int cps) {
  VLay L{};
  L.NP = D / 64;
  const int nqb = cps == 2 ? QBufsOf<2>::n : QBufsOf<1>::n;
  const int q_rows = NQ < 8 ? 8 : (NQ + 7) & ~7;
  L.q_panel = uint32_t(q_rows) * 128;
  L.q_buf = uint32_t(L.NP) * L.q_panel;
  L.ring_off = (uint32_t(nqb) * L.q_buf + 1023u) & ~1023u;
  L.kv_panel = uint32_t(TK) * 128;
  L.half_bytes = uint32_t(L.NP) * L.kv_panel;
  L.stage_bytes = 2 * L.half_bytes;
  L.nst = cps == 2 ? (D == 128 ? StagesOf<128, 2>::n : StagesOf<64, 2>::n)
                   : (D == 128 ? StagesOf<128, 1>::n : StagesOf<64, 1>::n);
  L.mask_off = L.ring_off + uint32_t(L.nst) * L.stage_bytes;
  L.bar_off = L.mask_off + ((uint32_t(L.nst) * kLoaders + 7u) & ~7u);
  L.misc_off = L.bar_off + uint32_t(2 * L.nst + 4 + 2 * nqb + 2) * 8;
  L.total = L.misc_off + 16 + 1024;
  return L;
}

// CTA that owns flattened tile x, for start(c) = c * total / G.
__device__ __forceinline__ int cta_of(long long x, long long total, int G) {
  return int(((x + 1) * G + total - 1) / total) - 1;
}

// One stream-K segment of this CTA: tiles [ta, ta + n) of unit u.
struct Seg {
  int u, ta, n;
};
__device__ __forceinline__ Seg next_seg(long long& t, long long t1, int tiles_u) {
  Seg s;
  s.u = int(t / tiles_u);
  s.ta = int(t % tiles_u);
  const long long rem_t = t1 - t;
  const int tb = int(rem_t < (long long)(tiles_u - s.ta) ? s.ta + rem_t : tiles_u);
  s.n = tb - s.ta;
  t += s.n;
  return s;
}

// M: rows of the S and P V MMAs, 64 when the query rows fit (they then spread
// over the four lane quarters, 16 each), else 128 (one row per lane).
// CPS: CTAs resident per SM (2 only with M = 64: 72 registers a thread, 256
// tensor-memory columns, one query buffer and fewer stages each).
template <int D, int M, int CPS>
__global__ void __launch_bounds__(NTH, CPS) verify_kernel(const __grid_constant__ VerifyArgs A) {
  static_assert(M == 64 || M == 128, "MMA rows");
  static_assert(CPS == 1 || (CPS == 2 && M == 64), "two CTAs per SM only with 64-row MMAs");
  using Tm = TmemCfg<D, CPS>;
  const VLay& Ly = A.lay;
  constexpr int NSTAGE = StagesOf<D, CPS>::n;   // == A.lay.nst
  constexpr int NQB = QBufsOf<CPS>::n;          // query buffers
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint8_t* masks = smem + Ly.mask_off;   // [NSTAGE][kLoaders]: valid-key bits, kKpw per byte
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Ly.bar_off);
  uint64_t* empty = full + NSTAGE;
  uint64_t* s_full = empty + NSTAGE;
  uint64_t* p_full = s_full + 2;
  uint64_t* q_full = p_full + 2;
  uint64_t* q_empty = q_full + NQB;
  uint64_t* mma_done = q_empty + NQB;    // the S issuer's MMAs have completed
  uint64_t* pv_done = mma_done + 1;      // the P V issuer's MMAs have completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly.misc_off + 8);
  int* q_hi = reinterpret_cast<int*>(smem + Ly.misc_off + 12);   // query loads issued: [0, q_hi)

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int T = A.T, NQ = A.NQ, GQ = A.G;
  const int n_act = M == 64 ? (NQ + 15) >> 4 : (NQ + 31) >> 5;   // softmax warps holding query rows
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 32 * kLoaders + kLoaders);
      mbar_init(&empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 32 * n_act);
    }
    for (int x = 0; x < NQB; ++x) {
      mbar_init(&q_full[x], 1);
      mbar_init(&q_empty[x], 1);
    }
    mbar_init(mma_done, 1);
    mbar_init(pv_done, 1);
    *abort_flag = 0;
    *q_hi = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "n"(Tm::cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  pdl_launch_dependents();
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int G = gridDim.x;
  const long long total = A.total;
  const long long t0 = (long long)blockIdx.x * total / G;
  const long long t1 = (long long)(blockIdx.x + 1) * total / G;
  const int tiles_u = A.tiles_u, ctx_tiles = A.ctx_tiles;
  const int units_per_layer = A.B * A.hkv;

  if (warp >= kLoaderWarp0 && warp < kLoaderWarp0 + kLoaders) {
    // =============================================================== loaders
    // Loader warp lw fetches keys [8 lw, 8 lw + 8) of every tile: lane l holds
    // the index of key 8 lw + l % 8, then the warp copies the K and V rows of
    // its keys with 16-byte cp.async (one row of 256 bytes per half-warp at
    // d = 128) straight into the 128-byte-swizzled layout the MMA reads;
    // unused rows are zero-filled.  Each thread's copies arrive on the stage's barrier as
    // they complete (cp.async.mbarrier.arrive), and lane 0 arrives once more
    // after publishing the warp's valid-key bits.
    const int lw = warp - kLoaderWarp0;
    constexpr int CH = D / 8;             // 16-byte chunks per row
    constexpr int KPI = 32 / CH;          // rows per warp instruction
    constexpr int NI = kKpw / KPI;        // instructions per tensor
    const int c = lane % CH;
    const int ksub = lane / CH;
    int gi = 0;
    int s = 0;
    bool live = true;     // false once a wait gave up
    const int kk = kKpw * lw + (lane % kKpw);   // key whose index this lane reads
    // The I_verify entry of key kk is loaded one tile ahead, so that a tile's
    // copies do not wait for its index to come back from memory.  The walk
    // over (sequence, KV head, tile) of the prefetched tile advances by
    // increments (no division on the loaders' path).
    long long tp = t0;
    int ptt = int(t0 % tiles_u), pg, pb;
    {
      const int pu = int(t0 / tiles_u);
      pg = pu % A.hkv;
      pb = (pu % units_per_layer) / A.hkv;
    }
    auto fetch_index = [&]() -> int {
      int v = -1;
      if (!A.dense && tp < t1 && ptt < ctx_tiles) {
        const int jj = ptt * TK + kk;
        if (jj < A.k) v = __ldg(A.ivf + size_t(pb) * A.k + jj);
      }
      ++tp;
      if (++ptt == tiles_u) {
        ptt = 0;
        if (++pg == A.hkv) {
          pg = 0;
          if (++pb == A.B) pb = 0;
        }
      }
      return v;
    };
    int raw_next = fetch_index();
    uint32_t tmask = 0;   // bit j: tile gi - 1 - j came by TMA boxes
    for (long long t = t0; t < t1 && live; ++s) {
      const Seg sg = next_seg(t, t1, tiles_u);
      const int layer = sg.u / units_per_layer;
      const int b = (sg.u % units_per_layer) / A.hkv;
      const int g = sg.u % A.hkv;
      const VerifyLayerDev& Lr = A.layer[layer];
      int L = A.seq_len[b];
      if (L < 0 || L > A.Lcap) {
        if (lw == 0 && lane == 0 && g == 0 && layer == 0 && sg.ta == 0)
          flag_error(A.err, DUSTIN_DEV_SEQLEN);
        L = 0;
      }
      // this segment's query rows -> query buffer s % NQB, once the MMAs of the
      // segment that used it last are done
      const int qb = s % NQB;
      if (s % kLoaders == lw) {
        bool ok = true;
        if (lane == 0) {
          if (s >= NQB) ok = mbar_wait(&q_empty[qb], uint32_t(s / NQB - 1) & 1u, A.err, abort_flag);
          if (ok) {
            mbar_arrive_expect_tx(&q_full[qb], uint32_t(NQ) * D * 2);
#pragma unroll
            for (int h = 0; h < Ly.NP; ++h)
              tma_load_3d(sbase + uint32_t(qb * Ly.q_buf + h * Ly.q_panel), &A.qmap[layer], h * 64,
                          g * GQ, b * T, &q_full[qb]);
            atomicMax(q_hi, s + 1);
          }
        }
        if (!__shfl_sync(0xffffffffu, int(ok), 0)) break;
      }
      const uint16_t* kbase = Lr.k + size_t(b) * Lr.ksb + size_t(g) * Lr.ksh;
      const uint16_t* vbase = Lr.v + size_t(b) * Lr.vsb + size_t(g) * Lr.vsh;
      const size_t blk_off = (size_t(b) * A.hkv + g) * T * D;
      for (int i = 0; i < sg.n; ++i, ++gi) {
        const int tt = sg.ta + i;
        const bool blk = tt >= ctx_tiles;
        int raw = raw_next;                      // this tile's index (sparse context tiles)
        raw_next = fetch_index();
        if (blk) raw = kk;
        else if (A.dense) raw = tt * TK + kk;
        const int st = int(gi % NSTAGE);
        if (gi >= NSTAGE &&
            !__all_sync(0xffffffffu, mbar_wait(&empty[st], uint32_t(gi / NSTAGE - 1) & 1u, A.err, abort_flag))) {
          live = false;
          break;
        }
        // a dense context tile wholly inside the sequence: TMA boxes, issued by
        // one lane, the byte count armed with that lane's arrival (the other
        // threads arrive as for a gathered tile, with nothing in flight)
        const bool by_tma = A.tma && !blk && (tt + 1) * TK <= L;
        tmask = (tmask << 1) | uint32_t(by_tma);
        if (by_tma) {
          const uint32_t stage = sbase + uint32_t(Ly.ring_off + size_t(st) * Ly.stage_bytes);
          if (lane == 0) masks[st * kLoaders + lw] = uint8_t((1u << kKpw) - 1u);
          if (lw == 0 && lane == 0) {
            mbar_arrive_expect_tx(&full[st], uint32_t(2 * TK * D * 2));
            const uint64_t pol = policy_evict_first();
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
              const uint32_t dk = stage + uint32_t(h * Ly.kv_panel);
              const uint32_t dv = dk + uint32_t(Ly.half_bytes);
              if (A.kvrank[layer] == 2) {
                const int row = (b * A.hkv + g) * A.Lcap + tt * TK;
                tma_load_2d_u32(dk, &A.kmap[layer], h * 64, row, &full[st], pol);
                tma_load_2d_u32(dv, &A.vmap[layer], h * 64, row, &full[st], pol);
              } else {
                tma_load_4d_u32(dk, &A.kmap[layer], h * 64, tt * TK, g, b, &full[st], pol);
                tma_load_4d_u32(dv, &A.vmap[layer], h * 64, tt * TK, g, b, &full[st], pol);
              }
            }
          } else if (lane == 0) {
            mbar_arrive(&full[st]);
          }
          cp_async_arrive_noinc(&full[st]);
          continue;
        }
        bool valid;
        if (blk) valid = raw < T;
        else if (A.dense) valid = raw < L;
        else {
          valid = raw >= 0 && raw < L;
          if (lane < kKpw && (raw < -1 || raw >= L)) flag_error(A.err, DUSTIN_DEV_INDEX);
        }
        const uint32_t vbits = __ballot_sync(0xffffffffu, valid) & ((1u << kKpw) - 1u);
        const uint32_t stage = sbase + uint32_t(Ly.ring_off + size_t(st) * Ly.stage_bytes);
#pragma unroll
        for (int m = 0; m < 2 * NI; ++m) {
          const int which = m / NI;
          const int kl = (m % NI) * KPI + ksub;            // key within the warp's 16
          const int r = __shfl_sync(0xffffffffu, raw, kl);
          const bool ok = (vbits >> kl) & 1u;
          const int rr = ok ? r : 0;
          const uint16_t* src;
          if (blk) src = (which ? Lr.vb : Lr.kb) + blk_off + size_t(rr) * D + c * 8;
          else if (which) src = vbase + size_t(rr) * Lr.vsl + c * 8;
          else src = kbase + size_t(rr) * Lr.ksl + c * 8;
          const int key = kKpw * lw + kl;
          cp_async16(stage + uint32_t(which * Ly.half_bytes + (c >> 3) * Ly.kv_panel) + swz(key, c & 7),
                     src, ok ? 16u : 0u);
        }
        if (lane == 0) masks[st * kLoaders + lw] = uint8_t(vbits);
        cp_async_arrive_noinc(&full[st]);
        if (lane == 0) mbar_arrive(&full[st]);
      }
    }
    cp_async_wait_all();
    // the boxes this lane issued for the last NSTAGE tiles have landed (each
    // is the latest phase of its stage) before the CTA may exit
    if (lw == 0 && lane == 0)
      for (int j = 0; j < NSTAGE && j < gi; ++j)
        if ((tmask >> j) & 1u)
          mbar_drain(&full[(gi - 1 - j) % NSTAGE], uint32_t((gi - 1 - j) / NSTAGE) & 1u, A.err);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ================================================================ S MMAs
    // S = Q K^T of tile g into S buffer g % 2, once its rows have landed and
    // the softmax has read that buffer's previous tile (g - 2); with P stored
    // over S, once P V of tile g - 2 has read that P
    if (lane == 0) {
      constexpr uint32_t kIdS = tc_idesc(M, TK, 0);
      int gi = 0;
      int s = 0;
      bool issued = false;
      bool live = true;   // false once a wait gave up: issue nothing more
      for (long long t = t0; t < t1 && live; ++s) {
        const Seg sg = next_seg(t, t1, tiles_u);
        const int qb = s % NQB;
        const uint32_t qbuf = sbase + uint32_t(qb * Ly.q_buf);
        if (!mbar_wait(&q_full[qb], uint32_t(s / NQB) & 1u, A.err, abort_flag)) break;
        for (int i = 0; i < sg.n; ++i, ++gi) {
          const int st = int(gi % NSTAGE);
          if ((gi >= 2 && !(CPS == 2 ? mbar_wait(&empty[(gi - 2) % NSTAGE], uint32_t((gi - 2) / NSTAGE) & 1u,
                                                   A.err, abort_flag)
                                     : mbar_wait(&p_full[gi & 1], uint32_t((gi >> 1) - 1) & 1u, A.err,
                                                 abort_flag))) ||
              !mbar_wait(&full[st], uint32_t(gi / NSTAGE) & 1u, A.err, abort_flag)) {
            live = false;
            break;
          }
          issued = true;
          fence_proxy_async();   // the rows were written by cp.async (generic proxy)
          tc_fence_after();
          const uint32_t kst = sbase + uint32_t(Ly.ring_off + size_t(st) * Ly.stage_bytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = uint32_t((kk & 3) * 32);
            const uint64_t a = tc_desc(qbuf + uint32_t((kk >> 2) * Ly.q_panel) + koff, 16, 1024);
            const uint64_t bd = tc_desc(kst + uint32_t((kk >> 2) * Ly.kv_panel) + koff, 16, 1024);
            tc_mma_ss(tmem + uint32_t(kSCol + (gi & 1) * TK), a, bd, kIdS, kk > 0);
          }
          tc_commit(&s_full[gi & 1]);
        }
        if (live) tc_commit(&q_empty[qb]);   // the segment's query rows are no longer read
      }
      // every MMA this thread issued has completed before tensor memory is freed
      if (issued) {
        tc_commit(mma_done);
        mbar_drain(mma_done, 0, A.err);
      }
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ============================================================== P V MMAs
    // O (+)= P V of tile g once the softmax has stored P (the first tile of a
    // segment overwrites O, which the softmax read for the previous segment
    // before it stored that P); the commit frees the tile's stage
    if (lane == 0) {
      constexpr uint32_t kIdPV = tc_idesc(M, D, 1);
      const uint32_t o_tmem = tmem + Tm::o_col;
      int gi = 0;
      bool issued = false;
      bool live = true;
      for (long long t = t0; t < t1 && live;) {
        const Seg sg = next_seg(t, t1, tiles_u);
        for (int i = 0; i < sg.n; ++i, ++gi) {
          if (!mbar_wait(&p_full[gi & 1], uint32_t(gi >> 1) & 1u, A.err, abort_flag)) {
            live = false;
            break;
          }
          issued = true;
          tc_fence_after();
          const int st = int(gi % NSTAGE);
          const uint32_t vst =
              sbase + uint32_t(Ly.ring_off + size_t(st) * Ly.stage_bytes + Ly.half_bytes);
          const uint32_t p_tmem = tmem + uint32_t(Tm::p_col + (gi & 1) * Tm::p_stride);
#pragma unroll
          for (int kk = 0; kk < TK / 16; ++kk) {
            const uint64_t bd = tc_desc(vst + uint32_t(kk * 2048), uint32_t(Ly.kv_panel), 1024);
            tc_mma_ts(o_tmem, p_tmem + uint32_t(kk * 8), bd, kIdPV, (i > 0 || kk > 0) ? 1 : 0);
          }
          tc_commit(&empty[st]);   // S and P V of tile gi done: its stage is free
        }
      }
      if (issued) {
        tc_commit(pv_done);
        mbar_drain(pv_done, 0, A.err);
      }
    }
    __syncwarp();
  } else if (warp < n_act) {
    if constexpr (M == 64) {
      // ====================================================== softmax (M = 64)
      // Warp w holds query rows 16 w .. 16 w + 15 (lanes 32 w .. 32 w + 15).
      // Thread t takes rows r0 = 16 w + t / 4 and r1 = r0 + 8 and, of each, the
      // keys 8 c + 2 (t % 4) + {0, 1} of the eight 8-key chunks c (16x256b
      // loads).  The four threads of a quad share their rows' maxima by
      // shuffles and keep partial row sums, added up in the epilogue.  P goes
      // back with the 16x128b shape, whose column t % 4 of each 4-column chunk
      // is exactly this thread's bf16 pair of keys.
      const int q4 = lane & 3;
      const int r0 = 16 * warp + (lane >> 2), r1 = r0 + 8;
      const bool act0 = r0 < NQ, act1 = r1 < NQ;
      const int tq0 = act0 ? r0 / GQ : 0, tq1 = act1 ? r1 / GQ : 0;
      const float scale = A.scale_log2;
      const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
      const uint32_t o_lane = lane_base + uint32_t(Tm::o_col);
      int gi = 0;
      bool live = true;   // false once a wait gave up (warp-uniform)
      for (long long t = t0; t < t1 && live;) {
        const Seg sg = next_seg(t, t1, tiles_u);
        const int u = sg.u, n = sg.n;
        const int layer = u / units_per_layer;
        const int b = (u % units_per_layer) / A.hkv;
        const int g = u % A.hkv;
        const VerifyLayerDev& Lr = A.layer[layer];
        float mref0 = -INFINITY, mref1 = -INFINITY;   // reference maxima (log2 domain)
        float lsum0 = 0.f, lsum1 = 0.f;               // this thread's share of the row sums
        for (int i = 0; i < n; ++i, ++gi) {
          const int st = int(gi % NSTAGE);
          if (!__all_sync(0xffffffffu, mbar_wait(&full[st], uint32_t(gi / NSTAGE) & 1u, A.err, abort_flag) &&
                                           mbar_wait(&s_full[gi & 1], uint32_t(gi >> 1) & 1u, A.err, abort_flag))) {
            live = false;
            break;
          }
          const unsigned long long mw = *reinterpret_cast<const unsigned long long*>(masks + st * kLoaders);
          const bool blk = sg.ta + i >= ctx_tiles;
          tc_fence_after();
          float x0[16], x1[16];   // scores of rows r0, r1: entry 2 c + e is key 8 c + 2 q4 + e
          {
            uint32_t sv[32];
            tc_ld16x256_x8(lane_base + uint32_t(kSCol + (gi & 1) * TK), sv);
  #pragma unroll
            for (int c = 0; c < 8; ++c) {
              x0[2 * c] = __uint_as_float(sv[4 * c]);
              x0[2 * c + 1] = __uint_as_float(sv[4 * c + 1]);
              x1[2 * c] = __uint_as_float(sv[4 * c + 2]);
              x1[2 * c + 1] = __uint_as_float(sv[4 * c + 3]);
            }
          }
          if (blk || mw != ~0ull) {
            // keys the tile does not use (and, in the block tile, u > t) get -inf
  #pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int key = 8 * (j >> 1) + 2 * q4 + (j & 1);
              const bool v = ((mw >> key) & 1ull) != 0;
              x0[j] = v && (!blk || key <= tq0) ? x0[j] : -INFINITY;
              x1[j] = v && (!blk || key <= tq1) ? x1[j] : -INFINITY;
            }
          }
          float m0 = x0[0], m1 = x1[0];
  #pragma unroll
          for (int j = 1; j < 16; ++j) {
            m0 = fmaxf(m0, x0[j]);
            m1 = fmaxf(m1, x1[j]);
          }
          m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
          m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
          m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
          m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
          // (a row past NQ takes -inf as its max: it never rescales O, and its
          // P and O rows are never read)
          const float mx0 = act0 ? m0 * scale : -INFINITY, mx1 = act1 ? m1 * scale : -INFINITY;
          float alpha0 = 1.f, alpha1 = 1.f;
          if (mx0 > mref0 + 8.f) {
            alpha0 = fast_exp2(mref0 - mx0);
            mref0 = mx0;
            lsum0 *= alpha0;
          }
          if (mx1 > mref1 + 8.f) {
            alpha1 = fast_exp2(mref1 - mx1);
            mref1 = mx1;
            lsum1 *= alpha1;
          }
          const float nb0 = (mref0 == -INFINITY) ? 0.f : -mref0;
          const float nb1 = (mref1 == -INFINITY) ? 0.f : -mref1;
          uint32_t pk[16];   // 16x128b order: pk[2 c] row r0, pk[2 c + 1] row r1
          float la[2] = {0.f, 0.f}, lb[2] = {0.f, 0.f};
  #pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t v0 = pack_bf16(fast_exp2(fmaf(x0[2 * c], scale, nb0)), fast_exp2(fmaf(x0[2 * c + 1], scale, nb0)));
            const uint32_t v1 = pack_bf16(fast_exp2(fmaf(x1[2 * c], scale, nb1)), fast_exp2(fmaf(x1[2 * c + 1], scale, nb1)));
            pk[2 * c] = v0;
            pk[2 * c + 1] = v1;
            la[c & 1] += __uint_as_float(v0 << 16) + __uint_as_float(v0 & 0xFFFF0000u);
            lb[c & 1] += __uint_as_float(v1 << 16) + __uint_as_float(v1 & 0xFFFF0000u);
          }
          lsum0 += la[0] + la[1];
          lsum1 += lb[0] + lb[1];
          // rescale this thread's O rows once P V of the previous tile is in
          if (i > 0 && __any_sync(0xffffffffu, alpha0 != 1.f || alpha1 != 1.f)) {
            if (!__all_sync(0xffffffffu, mbar_wait(&empty[(gi - 1) % NSTAGE], uint32_t((gi - 1) / NSTAGE) & 1u,
                                                   A.err, abort_flag))) {
              live = false;
              break;
            }
            tc_fence_after();
  #pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t o[16];
              tc_ld16x256_x4(o_lane + uint32_t(c), o);
  #pragma unroll
              for (int x = 0; x < 16; ++x)
                o[x] = __float_as_uint(__uint_as_float(o[x]) * ((x & 2) ? alpha1 : alpha0));
              tc_st16x256_x4(o_lane + uint32_t(c), o);
            }
          }
          // P buffer gi % 2 is free once P V of tile gi - 2 has completed (when
          // P is stored over S, S of tile gi was issued only after that)
          if (CPS == 1 && gi >= 2 &&
              !__all_sync(0xffffffffu, mbar_wait(&empty[(gi - 2) % NSTAGE], uint32_t((gi - 2) / NSTAGE) & 1u,
                                                 A.err, abort_flag))) {
            live = false;
            break;
          }
          tc_st16x128_x8(lane_base + uint32_t(Tm::p_col + (gi & 1) * Tm::p_stride), pk);
          tc_fence_before();
          mbar_arrive(&p_full[gi & 1]);
        }

        if (!live) break;
        // ----------------------------------------------------------- epilogue
        lsum0 += __shfl_xor_sync(0xffffffffu, lsum0, 1);
        lsum1 += __shfl_xor_sync(0xffffffffu, lsum1, 1);
        lsum0 += __shfl_xor_sync(0xffffffffu, lsum0, 2);
        lsum1 += __shfl_xor_sync(0xffffffffu, lsum1, 2);
        const int seg_first = cta_of((long long)u * tiles_u, total, G);
        const int seg_last = cta_of((long long)u * tiles_u + tiles_u - 1, total, G);
        const int n_seg = seg_last - seg_first + 1;
        const int seg = blockIdx.x - seg_first;
        const size_t slot_floats = size_t(A.slot_floats);   // NQ*D + 2*NQ, rounded to 4
        float* part = A.partial + (size_t(u) * A.max_seg + seg) * slot_floats;
        if (!__all_sync(0xffffffffu, mbar_wait(&empty[(gi - 1) % NSTAGE], uint32_t((gi - 1) / NSTAGE) & 1u,
                                               A.err, abort_flag))) {
          live = false;
        } else {
          tc_fence_after();
          const int ra = act0 ? r0 : 0, rb = act1 ? r1 : 0;
          float* d0 = n_seg == 1 ? Lr.o + ((size_t(b) * T + ra / GQ) * A.hq + size_t(g) * GQ + ra % GQ) * D
                                 : part + size_t(ra) * D;
          float* d1 = n_seg == 1 ? Lr.o + ((size_t(b) * T + rb / GQ) * A.hq + size_t(g) * GQ + rb % GQ) * D
                                 : part + size_t(rb) * D;
          const float os0 = n_seg == 1 ? (lsum0 > 0.f ? 1.f / lsum0 : 0.f) : 1.f;
          const float os1 = n_seg == 1 ? (lsum1 > 0.f ? 1.f / lsum1 : 0.f) : 1.f;
  #pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t o[16];
            tc_ld16x256_x4(o_lane + uint32_t(c), o);   // collective: every lane loads
  #pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const int col = c + 8 * cc + 2 * q4;
              if (act0)
                *reinterpret_cast<float2*>(d0 + col) =
                    make_float2(__uint_as_float(o[4 * cc]) * os0, __uint_as_float(o[4 * cc + 1]) * os0);
              if (act1)
                *reinterpret_cast<float2*>(d1 + col) =
                    make_float2(__uint_as_float(o[4 * cc + 2]) * os1, __uint_as_float(o[4 * cc + 3]) * os1);
            }
          }
          if (n_seg > 1 && q4 == 0) {
            if (act0) {
              part[size_t(NQ) * D + r0] = mref0;
              part[size_t(NQ) * D + NQ + r0] = lsum0;
            }
            if (act1) {
              part[size_t(NQ) * D + r1] = mref1;
              part[size_t(NQ) * D + NQ + r1] = lsum1;
            }
          }
        }
        tc_fence_before();
      }
    } else {
      // =============================================================== softmax
      const int row = tid;             // query row == tensor-memory lane
      const bool active = row < NQ;
      const int tq_row = active ? row / GQ : 0;
      const float scale = A.scale_log2;
      const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
      const uint32_t o_lane = lane_base + uint32_t(Tm::o_col);
      int gi = 0;
      bool live = true;   // false once a wait gave up (warp-uniform)
      for (long long t = t0; t < t1 && live;) {
        const Seg sg = next_seg(t, t1, tiles_u);
        const int u = sg.u, n = sg.n;
        const int layer = u / units_per_layer;
        const int b = (u % units_per_layer) / A.hkv;
        const int g = u % A.hkv;
        const VerifyLayerDev& Lr = A.layer[layer];
        float mref = -INFINITY, lsum = 0.f;   // reference max (log2 domain) and row sum
        for (int i = 0; i < n; ++i, ++gi) {
          const int st = int(gi % NSTAGE);
          if (!__all_sync(0xffffffffu, mbar_wait(&full[st], uint32_t(gi / NSTAGE) & 1u, A.err, abort_flag) &&
                                           mbar_wait(&s_full[gi & 1], uint32_t(gi >> 1) & 1u, A.err, abort_flag))) {
            live = false;
            break;
          }
          const unsigned long long mw = *reinterpret_cast<const unsigned long long*>(masks + st * kLoaders);
          const bool blk = sg.ta + i >= ctx_tiles;
          tc_fence_after();
          float s[TK];
          tc_ld32(lane_base + uint32_t(kSCol + (gi & 1) * TK), reinterpret_cast<uint32_t*>(s));
          tc_ld32(lane_base + uint32_t(kSCol + (gi & 1) * TK + 32), reinterpret_cast<uint32_t*>(s + 32));
          if (blk || mw != ~0ull) {
            // rows the tile does not use (and, in the block tile, u > t) get -inf
  #pragma unroll
            for (int j = 0; j < TK; ++j) {
              const bool valid = ((mw >> j) & 1ull) != 0 && (!blk || j <= tq_row);
              s[j] = valid ? s[j] : -INFINITY;
            }
          }
          // raw row max (the scale is positive)
          float m8[8];
  #pragma unroll
          for (int x = 0; x < 8; ++x)
            m8[x] = fmaxf(fmaxf(fmaxf(s[x], s[x + 8]), fmaxf(s[x + 16], s[x + 24])),
                          fmaxf(fmaxf(s[x + 32], s[x + 40]), fmaxf(s[x + 48], s[x + 56])));
          // (a query row past NQ has an S row computed from whatever lies past
          // the query rows: its max is taken as -inf, so it never rescales O;
          // its P and O rows are never read)
          const float mx = active ? fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                          fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * scale
                                  : -INFINITY;
          float alpha = 1.f;
          if (mx > mref + 8.f) {   // also the first tile with a valid key
            alpha = fast_exp2(mref - mx);   // 0 while mref is -inf
            mref = mx;
            lsum *= alpha;
          }
          const float nb = (mref == -INFINITY) ? 0.f : -mref;
          uint32_t pk[TK / 2];
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
  #pragma unroll
          for (int j = 0; j < TK; j += 2) {
            const uint32_t v = pack_bf16(fast_exp2(fmaf(s[j], scale, nb)), fast_exp2(fmaf(s[j + 1], scale, nb)));
            pk[j / 2] = v;
            ls[(j >> 1) & 3] += __uint_as_float(v << 16) + __uint_as_float(v & 0xFFFF0000u);
          }
          lsum += (ls[0] + ls[1]) + (ls[2] + ls[3]);
          // rescale this row of O once P V of the previous tile is in (the
          // first tile of a segment overwrites O); tensor-memory loads and
          // stores are collective, so the whole warp takes part
          if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
            if (!__all_sync(0xffffffffu, mbar_wait(&empty[(gi - 1) % NSTAGE], uint32_t((gi - 1) / NSTAGE) & 1u,
                                                   A.err, abort_flag))) {
              live = false;
              break;
            }
            tc_fence_after();
  #pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t o[32];
              tc_ld32(o_lane + uint32_t(c), o);
  #pragma unroll
              for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
              tc_st32(o_lane + uint32_t(c), o);
            }
          }
          // P buffer gi % 2 is free once P V of tile gi - 2 has completed (the
          // two issuers' MMAs are not ordered with each other)
          if (gi >= 2 && !__all_sync(0xffffffffu, mbar_wait(&empty[(gi - 2) % NSTAGE],
                                                           uint32_t((gi - 2) / NSTAGE) & 1u, A.err,
                                                           abort_flag))) {
            live = false;
            break;
          }
          tc_st32(lane_base + uint32_t(Tm::p_col + (gi & 1) * Tm::p_stride), pk);
          tc_fence_before();
          mbar_arrive(&p_full[gi & 1]);
        }

        if (!live) break;
        // ----------------------------------------------------------- epilogue
        const int seg_first = cta_of((long long)u * tiles_u, total, G);
        const int seg_last = cta_of((long long)u * tiles_u + tiles_u - 1, total, G);
        const int n_seg = seg_last - seg_first + 1;
        const int seg = blockIdx.x - seg_first;
        const size_t slot_floats = size_t(A.slot_floats);   // NQ*D + 2*NQ, rounded to 4
        float* part = A.partial + (size_t(u) * A.max_seg + seg) * slot_floats;
        if (!__all_sync(0xffffffffu, mbar_wait(&empty[(gi - 1) % NSTAGE], uint32_t((gi - 1) / NSTAGE) & 1u,
                                               A.err, abort_flag))) {
          live = false;
        } else {
          tc_fence_after();
          const int tq = active ? row / GQ : 0, hl = active ? row - (row / GQ) * GQ : 0;
          float* dst = n_seg == 1 ? Lr.o + ((size_t(b) * T + tq) * A.hq + size_t(g) * GQ + hl) * D
                                  : part + size_t(active ? row : 0) * D;
          const float osc = n_seg == 1 ? (lsum > 0.f ? 1.f / lsum : 0.f) : 1.f;
  #pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tc_ld32(o_lane + uint32_t(c), o);   // collective: every lane loads
            if (active) {
  #pragma unroll
              for (int x = 0; x < 32; x += 4)
                *reinterpret_cast<float4*>(dst + c + x) =
                    make_float4(__uint_as_float(o[x]) * osc, __uint_as_float(o[x + 1]) * osc,
                                __uint_as_float(o[x + 2]) * osc, __uint_as_float(o[x + 3]) * osc);
            }
          }
          if (active && n_seg > 1) {
            part[size_t(NQ) * D + row] = mref;
            part[size_t(NQ) * D + NQ + row] = lsum;
          }
        }
        tc_fence_before();
      }
    }
  }

  // Every query load has been issued: the last NQB of them (each the latest
  // phase of its buffer) have landed before the CTA exits.  Older ones were
  // waited for by the MMA thread before the buffer was reloaded.
  __syncthreads();
  if (warp == kLoaderWarp0 && lane == 0) {
    const int hi = *q_hi;
    for (int x = hi - NQB < 0 ? 0 : hi - NQB; x < hi; ++x)
      mbar_drain(&q_full[x % NQB], uint32_t(x / NQB) & 1u, A.err);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(Tm::cols)
                 : "memory");
}
// Log-sum-exp merge of the segments of every unit that the stream-K split
// cut into more than one (a one-segment unit was written by its CTA).  One
// thread per output float4; the partials of a segment are (unnormalised O,
// log2-domain reference max m, row sum l) relative to that m.
constexpr int kCombineThreads = 128;

template <int D>
__global__ void __launch_bounds__(kCombineThreads) verify_combine_kernel(const __grid_constant__ VerifyCombineArgs C) {
  pdl_launch_dependents();
  // every CTA waits for the stream-K kernel before it leaves, so that this
  // kernel completes only after it (the next launch waits on this one)
  pdl_wait();
  const int u = blockIdx.y;
  const int seg_first = cta_of((long long)u * C.tiles_u, C.total, C.main_grid);
  const int seg_last = cta_of((long long)u * C.tiles_u + C.tiles_u - 1, C.total, C.main_grid);
  const int n_seg = seg_last - seg_first + 1;
  if (n_seg == 1) return;
  const int q = blockIdx.x * kCombineThreads + threadIdx.x;
  if (q >= C.NQ * (D / 4)) return;
  const int r = q / (D / 4), c4 = q - r * (D / 4);
  const size_t slot = size_t(C.slot_floats);
  const float* base0 = C.partial + size_t(u) * C.max_seg * slot;
  const size_t mo = size_t(C.NQ) * D;   // m at mo + r, l at mo + NQ + r
  // the (m, l, O) of up to four segments are loaded at once (one round trip
  // to memory), then merged; more segments are taken in further rounds
  float M = -INFINITY;
  float lsc = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int g0 = 0; g0 < n_seg; g0 += 4) {
    float mv[4], lv[4];
    float4 xv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      mv[u] = -INFINITY;
      lv[u] = 0.f;
      xv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g0 + u < n_seg) {
        const float* ps = base0 + size_t(g0 + u) * slot;
        mv[u] = __ldg(ps + mo + r);
        lv[u] = __ldg(ps + mo + C.NQ + r);
        xv[u] = __ldg(reinterpret_cast<const float4*>(ps + size_t(r) * D) + c4);
      }
    }
    float Mn = M;
#pragma unroll
    for (int u = 0; u < 4; ++u) Mn = fmaxf(Mn, mv[u]);
    const float bv = (Mn == -INFINITY) ? 0.f : Mn;
    // rescale what the earlier rounds merged to the new reference
    const float a = (M == -INFINITY) ? 0.f : exp2f(M - bv);
    lsc *= a;
    acc.x *= a;
    acc.y *= a;
    acc.z *= a;
    acc.w *= a;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = (mv[u] == -INFINITY) ? 0.f : exp2f(mv[u] - bv);
      lsc += w * lv[u];
      acc.x += w * xv[u].x;
      acc.y += w * xv[u].y;
      acc.z += w * xv[u].z;
      acc.w += w * xv[u].w;
    }
    M = Mn;
  }
  const float inv = lsc > 0.f ? 1.f / lsc : 0.f;
  const int layer = u / C.units_per_layer;
  const int b = (u % C.units_per_layer) / C.hkv;
  const int g = u % C.hkv;
  const int tq = r / C.G, hl = r - (r / C.G) * C.G;
  reinterpret_cast<float4*>(C.o[layer] + ((size_t(b) * C.T + tq) * C.hq + size_t(g) * C.G + hl) * D)[c4] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

template <int D, int M, int CPS>
cudaError_t launch_main(const VerifyArgs& a, const VerifyLaunch& pl, cudaStream_t stream) {
  auto kern = verify_kernel<D, M, CPS>;
  static const cudaError_t attr = [&] {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kVerifySmem));
    if (e == cudaSuccess && CPS > 1)   // room for CPS CTAs' shared memory
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               int(cudaSharedmemCarveoutMaxShared));
    return e;
  }();
  if (attr != cudaSuccess) return attr;
  return launch_pdl(kern, dim3(pl.grid), dim3(NTH), pl.smem, stream, a);
}

template <int D>
cudaError_t launch_t(const VerifyArgs& a, const VerifyLaunch& pl, cudaStream_t stream) {
  // 64-row MMAs while the query rows fit them (NQ <= 64), two CTAs per SM
  // when the plan found room for them
  cudaError_t e = pl.cps == 2  ? launch_main<D, 64, 2>(a, pl, stream)
                  : a.NQ <= 64 ? launch_main<D, 64, 1>(a, pl, stream)
                               : launch_main<D, 128, 1>(a, pl, stream);
  if (e != cudaSuccess) return e;
  VerifyCombineArgs c;
  c.NQ = a.NQ;
  c.T = a.T;
  c.hq = a.hq;
  c.hkv = a.hkv;
  c.G = a.G;
  c.units_per_layer = a.B * a.hkv;
  c.tiles_u = a.tiles_u;
  c.total = a.total;
  c.main_grid = pl.grid;
  c.max_seg = a.max_seg;
  c.slot_floats = a.slot_floats;
  c.partial = a.partial;
  for (int l = 0; l < DUSTIN_MAX_LAYERS; ++l) c.o[l] = l < a.n_layers ? a.layer[l].o : nullptr;
  const dim3 cgrid((a.NQ * (D / 4) + kCombineThreads - 1) / kCombineThreads, unsigned(pl.units));
  return launch_pdl(verify_combine_kernel<D>, cgrid, dim3(kCombineThreads), 0, stream, c);
}

}  // namespace

VerifyLaunch verify_plan(int D, int NQ, int nkeys_cap, int B, int hkv, int n_layers, int dense,
                         int num_sms) {
  (void)dense;
  VerifyLaunch pl{};
  pl.D = D;
  // two CTAs per SM when the query rows fit 64-row MMAs and two CTAs' shared
  // memory fits an SM
  const VLay lay2 = make_lay(D, NQ, 2);
  pl.cps = (NQ <= 64 && 2 * (size_t(lay2.total) + 1024) <= kSmemPerSm) ? 2 : 1;
  const VLay lay = pl.cps == 2 ? lay2 : make_lay(D, NQ, 1);
  pl.lay = lay;
  pl.NST = lay.nst;
  pl.ctx_tiles = (nkeys_cap + TK - 1) / TK;
  pl.tiles_u = pl.ctx_tiles + 1;
  pl.units = (long long)B * hkv * n_layers;
  pl.total = pl.units * pl.tiles_u;
  // persistent: cps CTAs per SM
  long long grid = (long long)pl.cps * (num_sms > 0 ? num_sms : 148);
  if (grid > kVerifyGridMax) grid = kVerifyGridMax;
  if (grid > pl.total) grid = pl.total;
  pl.grid = int(grid);
  // Partial slots per unit, bounded for any grid <= kVerifyGridMax: a unit of
  // tiles_u tiles meets at most tiles_u / per + 2 CTAs of >= per tiles each.
  const long long per = pl.total / kVerifyGridMax;
  pl.max_seg = int(pl.tiles_u / (per > 0 ? per : 1)) + 2;
  pl.slot_floats = ((long long)NQ * D + 2LL * NQ + 3) / 4 * 4;   // 16-byte aligned slots
  pl.smem = lay.total;
  return pl;
}

size_t verify_scratch_bytes(const VerifyLaunch& pl) {
  return size_t(pl.units) * pl.max_seg * size_t(pl.slot_floats) * 4;
}

cudaError_t verify_launch(const VerifyArgs& a, const VerifyLaunch& pl, cudaStream_t stream) {
  if (pl.D == 128) return launch_t<128>(a, pl, stream);
  if (pl.D == 64) return launch_t<64>(a, pl, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dustin
