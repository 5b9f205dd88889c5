// kda_tc.cu -- fused KDA chunked forward on the Blackwell tensor cores
// (tcgen05 + tensor memory + TMA), bf16 inputs, dk = dv = 128, 64-token
// chunks, fp32 state and accumulation.
//
// One CTA owns one (sequence, head, half of the value channels) and walks
// its sequence chunk by chunk; the two halves of a head run as independent
// CTAs (the intra-chunk work is repeated, the state work is split).  The
// state half S (128 key channels x 64 value channels, fp32) lives in tensor
// memory for the whole sequence.
//
// Per chunk (C = 64 rows r, key channel j, 16-token tiles a = r / 16):
//   alpha_r = max(1 / (1 + e^{x_r}), e^-5)   [= exp(max(-softplus(x), -5))]
//   E_r = prod of alpha from the start of r's tile to r      (in [e^-80, 1])
//   F_r = prod of alpha after r to the end of r's tile
//   P_a = product over tile a;   gamma_r = e^{G_r} = E_r prod_{c<a} P_c
// Gram matrices, column tile b (reference: cumulative decay at the end of
// tile b), rows r in tiles a >= b:
//   A_qk[r, i] = (q_r E_r m_ab) . (k_i F_i),  A_kk likewise with k_r, beta_r
//   m_aa = 1 / P_a (<= e^80),  m_ab = prod_{b<c<a} P_c for a > b (<= 1)
// so every factor stays inside the bf16/fp32 range: the 16-token bound on
// the cumulative log-decay (Kimi K3 architecture, orkas.ai, "A lower bound
// that erased a GPU code path") is what keeps m_aa below e^80, and lets the
// diagonal tiles go through the same dense product as the others.
// Then  T = (I + A_kk)^{-1}  (CUDA cores, fp32, blocked by 16x16 tiles),
//   W = T (beta K gamma),  U = T (beta V),  Delta = U - W S,
//   O = (Q gamma) S + A_qk Delta,  S <- gamma_C S + (K e^{G_C - G})^T Delta.
// The inter-chunk recurrence is serial over chunks (Towards AI walkthrough,
// "Infrastructure co-design": the chunk-to-chunk state dependency); the
// state stays on chip between chunks.
//
// Tensor-core products per chunk (M = 128 everywhere, bf16 operands in
// shared memory, fp32 accumulators in tensor memory):
//   Grams   4 x [128 x 16 x 128]   A_b (rows of tiles >= b) . Ktil_b^T
//   W^T     [128 x 64 x 64]        (beta K gamma)^T . T^T
//   U       [128 x 64 x 64]        [T; -] . (beta V)  (rows 64.. unused)
//   P       [128 x 64 x 128]       [W; Q gamma] . S   -> [W S; Q gamma S]
//   S      += [128 x 64 x 64]      (K dec)^T . Delta
//   O      += [128 x 64 x 64]      [-; A_qk] . Delta   (into P's lower rows)
#include <cudaTypedefs.h>
#include <stdio.h>

#include "kda_common.cuh"
#include "sm100.cuh"
#include "kda_tc_util.cuh"

namespace {

using namespace kda_tc;

constexpr int DK = 128, DV = 128, DVH = 64, C = 64;
constexpr int kThreads = 256;

// ---- shared memory map (bytes) ---------------------------------------------
// R0: TMA landing zone for one chunk (128B-swizzled rows of 64 channels)
constexpr int OFF_Q = 0;          // 2 x [64 rows][128 B]
constexpr int OFF_K = 16384;
constexpr int OFF_G = 32768;
constexpr int OFF_V = 49152;      // [64 rows][128 B] (this CTA's 64 value channels)
constexpr int R0_BYTES = 57344;
// R1: Gram operands, then (after the Gram products) the per-chunk scratch
constexpr int OFF_R1 = R0_BYTES;
constexpr int OFF_A1 = OFF_R1;                // [q0; k0; q1; k1] MN-major 128 x 128  32768
constexpr int OFF_B1 = OFF_A1 + 32768;        // [c0; c1]         MN-major  64 x 128  16384
constexpr int OFF_A2 = OFF_B1 + 16384;        // [q1'; k1']       MN-major  64 x 128  16384
constexpr int OFF_B2 = OFF_A2 + 16384;        // c0'              MN-major  32 x 128   8192
constexpr int R1_BYTES = 98304;
//   overlay after the Gram products:
constexpr int AKK_LD = 72;                        // fp32 row stride (floats)
constexpr int OFF_AKK = OFF_R1;                   // [64][72] fp32   18432
constexpr int OFF_TF = OFF_AKK + 18432;           // [64][72] fp32   18432
constexpr int OFF_T = OFF_TF + 18432;             // T bf16 K-major   8192
// [32][36] fp32 products of the block merges (4608 B), in the landing zone:
// the chunk's tiles have been read for the last time before the solve and
// the next chunk's are requested after it
constexpr int OFF_Y = OFF_Q;

// The rest of the map depends on the kernel mode: MODE 0 is the forward
// (state half: 64 value columns); MODE 1 is the segment summary, which
// carries the zero-start state half next to 64 columns of the segment's
// cumulative transition P (dk x dk), i.e. 128 state columns, and writes no
// output.  Lay<MODE> gives the offsets.
template <int MODE>
struct Lay {
  static constexpr int SC = MODE == 0 ? 64 : 128;          // state columns in TMEM
  static constexpr int OFF_SB = OFF_T + 8192;             // [S | P] bf16, MN-major 128 x SC
  static constexpr int OFF_DL = OFF_SB + SC * 256;         // Delta bf16, MN-major 64 x SC
  // rows 0..63 of the O product's A operand [-; A_qk] are never used: the
  // descriptor starts 8 KiB before A_qk, over Delta
  static constexpr int OFF_X = OFF_DL;                     // (MODE 0)
  static constexpr int OFF_AQ = OFF_DL + SC * 128;         // A_qk masked bf16 (MODE 0)
  static constexpr int OFF_BV = MODE == 0 ? OFF_AQ + 8192 : OFF_DL + SC * 128;  // (beta V)^T
  static constexpr int R1_BYTES_M = MODE == 0 ? R1_BYTES : OFF_BV + 8192 - OFF_R1;
  // R2: [W; Q gamma] MN-major, 128 M-rows x 128 K
  static constexpr int OFF_WQ = OFF_R1 + R1_BYTES_M;
  // R3: (beta K gamma)^T and (K dec)^T, K-major 128 x 64
  static constexpr int OFF_BKG = OFF_WQ + 32768;
  static constexpr int OFF_KD = OFF_BKG + 16384;
  // small
  static constexpr int OFF_BETA = OFF_KD + 16384;          // 64 bf16
  static constexpr int OFF_PT = OFF_BETA + 256;            // [4][128] fp32 tile products
  static constexpr int OFF_GC = OFF_PT + 2048;             // [128] fp32 gamma_C
  static constexpr int OFF_BAR = OFF_GC + 512;             // mbarriers
  static constexpr int OFF_MISC = OFF_BAR + 64;            // tmem base, abort flag
  static constexpr int SMEM_BYTES = OFF_MISC + 64;
  // TMEM columns
  static constexpr uint32_t TM_S = 0, TM_P = SC, TM_U = 2 * SC, TM_W = 2 * SC + 64,
                            TM_G = 2 * SC + 128;
};
static_assert(Lay<0>::OFF_BV + 8192 <= OFF_R1 + R1_BYTES, "R1 overlay");
static_assert(Lay<0>::SMEM_BYTES <= 232448 && Lay<1>::SMEM_BYTES <= 232448, "shared memory");
static_assert(Lay<1>::TM_G + 96 <= 512, "tensor memory");
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t TX_BYTES = 57344;  // Q, K, G (2 boxes each) + V (1 box)

#ifdef KDA_PHASE_TIMING
// cycles spent in each phase of the chunk loop by thread 0 of CTA (0, 0, 0)
__device__ unsigned long long kda_phase_cycles[24];
#define KDA_PHASE(k)                                                           \
  do {                                                                         \
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {   \
      const long long t_ = clock64();                                          \
      kda_phase_cycles[k] += (unsigned long long)(t_ - t_phase);               \
      t_phase = t_;                                                            \
    }                                                                          \
  } while (0)
#else
#define KDA_PHASE(k) do { } while (0)
#endif


struct TcParams {
  kda::FwdParams p;
  // debug dump of one (n, h): per chunk [64][.] fp32
  int dbg_n, dbg_h;
  float *dbg_gam, *dbg_aqk, *dbg_akk, *dbg_t, *dbg_w, *dbg_u;
};


// ---------------------------------------------------------------------------
template <int MODE, bool DBG>
__global__ void __launch_bounds__(kThreads, 1)
    kda_tc_fused_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_g,
                        const __grid_constant__ CUtensorMap tm_v, const TcParams tp) {
  extern __shared__ __align__(1024) unsigned char smem[];
  using Ly = Lay<MODE>;
  constexpr int SC = Ly::SC;
  constexpr int OFF_SB = Ly::OFF_SB, OFF_DL = Ly::OFF_DL, OFF_X = Ly::OFF_X, OFF_AQ = Ly::OFF_AQ;
  constexpr int OFF_BV = Ly::OFF_BV, OFF_WQ = Ly::OFF_WQ, OFF_BKG = Ly::OFF_BKG;
  constexpr int OFF_KD = Ly::OFF_KD, OFF_BETA = Ly::OFF_BETA, OFF_PT = Ly::OFF_PT;
  constexpr int OFF_GC = Ly::OFF_GC, OFF_BAR = Ly::OFF_BAR, OFF_MISC = Ly::OFF_MISC;
  constexpr uint32_t TM_S = Ly::TM_S, TM_P = Ly::TM_P, TM_U = Ly::TM_U, TM_W = Ly::TM_W;
  constexpr uint32_t TM_G = Ly::TM_G;
  const kda::FwdParams& p = tp.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = blockIdx.x, h = blockIdx.y;
  const int nseg = p.nseg > 1 ? p.nseg : 1;
  const int n = (int)blockIdx.z / nseg, sg = (int)blockIdx.z % nseg;  // sequence, segment
  const int H = p.H;

  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* bar_mma = bar_tma + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  int* s_abort = reinterpret_cast<int*>(smem + OFF_MISC + 4);
  unsigned short* s_beta_raw = reinterpret_cast<unsigned short*>(smem + OFF_BETA);
  auto beta_at = [&](int r) { return __uint_as_float((uint32_t)s_beta_raw[r] << 16); };
  float* s_pt = reinterpret_cast<float*>(smem + OFF_PT);
  float* s_gc = reinterpret_cast<float*>(smem + OFF_GC);
  float* s_akk = reinterpret_cast<float*>(smem + OFF_AKK);
  float* s_tf = reinterpret_cast<float*>(smem + OFF_TF);
  float* s_y = reinterpret_cast<float*>(smem + OFF_Y);

  int64_t row_base, t0, t1;
  if (!kda::seq_span(p, n, row_base, t0, t1)) return;  // uniform over the CTA
  if (nseg > 1) {  // this CTA's segment [t0 + sg * seglen, ...) of the sequence
    const int64_t a = t0 + (int64_t)sg * p.seglen;
    const int64_t b = a + p.seglen;
    t0 = a < t1 ? a : t1;
    t1 = b < t1 ? b : t1;
  }

  if (warp == 0) {
    sm100::tmem_alloc(s_tmem, TM_COLS);
    sm100::tmem_relinquish();
  }
  if (tid == 32) {
    sm100::mbar_init(bar_tma, 1);
    sm100::mbar_init(bar_mma, 1);
    sm100::fence_mbar_init();
    if (t1 > t0) {
      sm100::tma_prefetch_desc(&tm_q);
      sm100::tma_prefetch_desc(&tm_k);
      sm100::tma_prefetch_desc(&tm_g);
      sm100::tma_prefetch_desc(&tm_v);
    }
  }
  if (tid == 0) *s_abort = 0;
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_q = 32u * (warp & 3);  // this warp's TMEM lane quarter
  const int64_t sbase = ((int64_t)n * H + h) * (int64_t)DK * DV + half * DVH;
  // segment-indexed state slot [n][sg][h] of the segment scratch
  const int64_t segbase = (((int64_t)n * nseg + sg) * H + h) * (int64_t)DK * DV + half * DVH;

  // ---- initial state into TMEM (lane = key channel) ------------------------
  //   MODE 0: init_state (first segment) or the segment's resolved entry
  //   state; MODE 1: zero state and, in columns 64.., this half's columns of
  //   the identity (the transition of an empty prefix)
  if (warp < 4) {
    const int i = warp * 32 + lane;
    const float* src = nullptr;
    int64_t base = 0;
    if (MODE == 0) {
      if (sg == 0) { src = p.init_state; base = sbase; }
      else { src = p.seg_init; base = segbase; }
    }
    for (int c = 0; c < SC; c += 16) {
      uint32_t r[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float x = 0.0f;
        if (MODE == 0) {
          if (src) x = src[base + (int64_t)i * DV + c + e];
        } else if (c >= 64) {
          x = (i == half * 64 + (c - 64) + e) ? 1.0f : 0.0f;
        }
        r[e] = __float_as_uint(x);
      }
      sm100::tmem_st16(sm100::taddr(tmem, lane_q, TM_S + c), r);
    }
    sm100::tmem_wait_st();
  }

  const int64_t nchunks = (t1 - t0 + C - 1) / C;
  uint32_t mma_phase = 0;
  bool mma_inflight = false;
  bool tma_pending = nchunks > 0;  // a load into the landing zone is in flight
  uint32_t tma_parity = 0;
  auto issue_tma = [&](int64_t ci) {
    const int row = (int)(row_base + t0 + ci * C);
    sm100::mbar_arrive_expect_tx(bar_tma, TX_BYTES);
    sm100::tma_load_3d(smem + OFF_Q, &tm_q, bar_tma, 0, h, row);
    sm100::tma_load_3d(smem + OFF_Q + 8192, &tm_q, bar_tma, 64, h, row);
    sm100::tma_load_3d(smem + OFF_K, &tm_k, bar_tma, 0, h, row);
    sm100::tma_load_3d(smem + OFF_K + 8192, &tm_k, bar_tma, 64, h, row);
    sm100::tma_load_3d(smem + OFF_G, &tm_g, bar_tma, 0, h, row);
    sm100::tma_load_3d(smem + OFF_G + 8192, &tm_g, bar_tma, 64, h, row);
    sm100::tma_load_3d(smem + OFF_V, &tm_v, bar_tma, half * DVH, h, row);
  };
  // wait for the MMA batch just committed; records a timeout
  auto wait_mma = [&]() {
    const bool ok = sm100::mbar_wait(bar_mma, mma_phase & 1);
    if (ok) ++mma_phase;
    mma_inflight = !ok;
    if (!ok) {
      *s_abort = 1;
      if (p.dev_status) atomicExch(p.dev_status, (int32_t)KDA_ERR_TIMEOUT);
    }
    sm100::tc_fence_after();
  };
  auto commit_mma = [&]() { sm100::mma_commit(bar_mma); };
  auto sync_all = [&]() {
    sm100::tc_fence_before();
    __syncthreads();
    sm100::tc_fence_after();
  };

  // beta of row `tid` of the next chunk, kept as raw bf16 bits so that the
  // load is only waited for one chunk later
  const unsigned short* beta_g = static_cast<const unsigned short*>(p.beta);
  unsigned short beta_next = 0;
  if (tid < C && nchunks > 0 && t0 + tid < t1) beta_next = beta_g[(row_base + t0 + tid) * H + h];
  if (tid == 0 && nchunks > 0) issue_tma(0);

  // decay factors alpha of this thread's 32 rows (key channel tid & 127,
  // rows 32 * (tid >> 7) ..) for the chunk being prepared, and the tile
  // products of those rows into s_pt
  float al[32];
  auto gate_alpha = [&](int64_t cj) {
    const int j = tid & 127, pr = tid >> 7, jc = j & 63;
    const int64_t csj = t0 + cj * C;
    const int Lj = (t1 - csj) < C ? (int)(t1 - csj) : C;
    const unsigned char* sg = smem + OFF_G + (j >> 6) * 8192;
#pragma unroll
    for (int s2 = 0; s2 < 32; ++s2) {
      const int r = 32 * pr + s2;
      al[s2] = (r < Lj) ? alpha_of(ld_bf16(sg, sw128_off(r, jc))) : 1.0f;
    }
    float Pt0 = 1.0f, Pt1 = 1.0f;
#pragma unroll
    for (int s2 = 0; s2 < 16; ++s2) { Pt0 *= al[s2]; Pt1 *= al[16 + s2]; }
    s_pt[(2 * pr) * 128 + j] = Pt0;
    s_pt[(2 * pr + 1) * 128 + j] = Pt1;
  };
  auto wait_tma = [&](int64_t cj) {
    const bool ok = sm100::mbar_wait(bar_tma, (uint32_t)(cj & 1));
    if (!ok) {
      *s_abort = 1;
      if (p.dev_status) atomicExch(p.dev_status, (int32_t)KDA_ERR_TIMEOUT);
    }
    tma_pending = !ok;
    tma_parity = (uint32_t)(cj & 1);
  };
#ifdef KDA_PHASE_TIMING
  long long t_phase = clock64();
#endif
  for (int64_t ci = 0; ci < nchunks; ++ci) {
    const int64_t cs = t0 + ci * C;
    const int L = (t1 - cs) < C ? (int)(t1 - cs) : C;
    // step dumps exist only in the test-hook instantiation
    const bool dbg_nh = DBG && tp.dbg_gam && n == tp.dbg_n && h == tp.dbg_h;
    const bool dbg = dbg_nh && half == 0;
    const int64_t dbo = ci * C;  // debug row offset

    // ---- (A) inputs of this chunk (beta was fetched one chunk ahead) -------
    if (tid < C) s_beta_raw[tid] = beta_next;  // bf16 bits; readers widen them
    if (ci == 0) {
      wait_tma(0);
      gate_alpha(0);  // later chunks: computed while the previous chunk's P runs
    }
    KDA_PHASE(11);
    const bool aborted = sync_aborted(s_abort);
    KDA_PHASE(0);
    if (aborted) break;

    // ---- (B) gate: one key channel j, one half (two tiles) per thread -------
    {
      const int j = tid & 127, pr = tid >> 7;  // rows 32pr .. 32pr+31
      const unsigned char* sq = smem + OFF_Q + (j >> 6) * 8192;
      const unsigned char* sk = smem + OFF_K + (j >> 6) * 8192;
      const int jc = j & 63;
      // alpha of these rows and the tile products were computed earlier
      // (gate_alpha); q and k of the 32 rows now
      float qv[32], kv[32];
#pragma unroll
      for (int s2 = 0; s2 < 32; ++s2) {
        const int r = 32 * pr + s2;
        const uint32_t o = sw128_off(r, jc);
        const bool ok = r < L;
        qv[s2] = ok ? ld_bf16(sq, o) * p.scale : 0.0f;
        kv[s2] = ok ? ld_bf16(sk, o) : 0.0f;
      }
      const float P0 = s_pt[j], P1 = s_pt[128 + j], P2 = s_pt[256 + j], P3 = s_pt[384 + j];
      if (pr == 0) s_gc[j] = P0 * P1 * P2 * P3;
      // tile products are >= e^-80, so their inverses stay below e^80
      const float invPa = __fdividef(1.0f, pr == 0 ? P0 : P2);   // first tile of the half
      const float invPb = __fdividef(1.0f, pr == 0 ? P1 : P3);   // second tile
      // per-tile constants (tt = 0, 1 for the two tiles of this half)
      //   pre: gamma offset prod_{c<a} P_c;  post: Kdec offset prod_{c>a} P_c
      const float pre0 = pr == 0 ? 1.0f : P0 * P1, pre1 = pr == 0 ? P0 : P0 * P1 * P2;
      const float post0 = pr == 0 ? P1 * P2 * P3 : P3, post1 = pr == 0 ? P2 * P3 : 1.0f;
      // E (within-tile prefix) and F (within-tile suffix) products
      float E[32], F[32];
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        float e = 1.0f, f = 1.0f;
#pragma unroll
        for (int s2 = 0; s2 < 16; ++s2) { e *= al[16 * tt + s2]; E[16 * tt + s2] = e; }
#pragma unroll
        for (int s2 = 15; s2 >= 0; --s2) { F[16 * tt + s2] = f; f *= al[16 * tt + s2]; }
      }
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {  // rows 8g8 .. 8g8+7 of the half
        const int tt = g8 >> 1;
        const int rr = 8 * g8;
        float qE[8], kE[8], kF[8], t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          qE[e] = qv[rr + e] * E[rr + e];
          kE[e] = kv[rr + e] * E[rr + e];
          kF[e] = kv[rr + e] * F[rr + e];
        }
        // Gram operands of the two-level scheme (reference points: end of
        // tile 0 for rows/columns of the first half, end of tile 2 for the
        // second half, end of tile 1 for the cross block):
        //   half 0: row e^{G_r - G_15}, col e^{G_15 - G_i}, cross col e^{G_31 - G_i}
        //   half 1: row e^{G_r - G_47}, col e^{G_47 - G_i}, cross row e^{G_r - G_31}
        // each a within-tile product times a per-tile constant, all within
        // [e^-80, e^80] for the pairs that are kept.
        const float rs = tt == 0 ? invPa : 1.0f;      // diagonal-half row factor
        const float cs = tt == 0 ? 1.0f : invPb;      // diagonal-half column factor
        if (pr == 0) {
          const float csm = tt == 0 ? P1 : 1.0f;      // cross column factor
#pragma unroll
          for (int e = 0; e < 8; ++e) t[e] = qE[e] * rs;
          st8_bf16(smem + OFF_A1 + mn_off(rr, j, 2048), t);
#pragma unroll
          for (int e = 0; e < 8; ++e) t[e] = kE[e] * rs;
          st8_bf16(smem + OFF_A1 + mn_off(32 + rr, j, 2048), t);
#pragma unroll
          for (int e = 0; e < 8; ++e) t[e] = kF[e] * cs;
          st8_bf16(smem + OFF_B1 + mn_off(rr, j, 1024), t);
#pragma unroll
          for (int e = 0; e < 8; ++e) t[e] = kF[e] * csm;
          st8_bf16(smem + OFF_B2 + mn_off(rr, j, 512), t);
        } else {
          const float rsm = tt == 0 ? 1.0f : P2;      // cross row factor
#pragma unroll
          for (int e = 0; e < 8; ++e) t[e] = qE[e] * rs;
          st8_bf16(smem + OFF_A1 + mn_off(64 + rr, j, 2048), t);
#pragma unroll
          for (int e = 0; e < 8; ++e) t[e] = kE[e] * rs;
          st8_bf16(smem + OFF_A1 + mn_off(96 + rr, j, 2048), t);
#pragma unroll
          for (int e = 0; e < 8; ++e) t[e] = qE[e] * rsm;
          st8_bf16(smem + OFF_A2 + mn_off(rr, j, 1024), t);
#pragma unroll
          for (int e = 0; e < 8; ++e) t[e] = kE[e] * rsm;
          st8_bf16(smem + OFF_A2 + mn_off(32 + rr, j, 1024), t);
#pragma unroll
          for (int e = 0; e < 8; ++e) t[e] = kF[e] * cs;
          st8_bf16(smem + OFF_B1 + mn_off(32 + rr, j, 1024), t);
        }
        const float pre = tt == 0 ? pre0 : pre1, post = tt == 0 ? post0 : post1;
        const int r0 = 32 * pr + rr;  // chunk row of this group
        // Q gamma into rows 64.. of [W; Q gamma] (the output needs it)
        if (MODE == 0) {
#pragma unroll
          for (int e = 0; e < 8; ++e) t[e] = qE[e] * pre;
          st8_bf16(smem + OFF_WQ + mn_off(64 + r0, j, 2048), t);
        }
        // (beta K gamma)^T, K-major [j][r]
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = beta_at(r0 + e) * kE[e] * pre;
        st8_bf16(smem + OFF_BKG + k64_off(j, r0), t);
        // (K e^{G_C - G})^T, K-major [j][r]
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = kF[e] * post;
        st8_bf16(smem + OFF_KD + k64_off(j, r0), t);
        if (dbg && tp.dbg_gam) {
#pragma unroll
          for (int e = 0; e < 8; ++e) tp.dbg_gam[(dbo + r0 + e) * DK + j] = E[rr + e] * pre;
        }
      }
    }
    sm100::fence_async_smem();
    sync_all();
    KDA_PHASE(1);

    // ---- (C) Gram products: diagonal halves (M=128, N=64) and the cross
    //      block (M=64, N=32), K = 128 key channels ---------------------------
    if (tid == 0) {
      const uint32_t id1 = sm100::idesc_bf16(128, 64, 1, 1);
      const uint32_t id2 = sm100::idesc_bf16(64, 32, 1, 1);
      const uint32_t a1 = sm100::smem_u32(smem + OFF_A1), b1 = sm100::smem_u32(smem + OFF_B1);
      const uint32_t a2 = sm100::smem_u32(smem + OFF_A2), b2 = sm100::smem_u32(smem + OFF_B2);
#pragma unroll
      for (int s2 = 0; s2 < DK / 16; ++s2)
        sm100::mma_ss(tmem + TM_G, sm100::smem_desc(a1 + s2 * 4096, 2048, 128),
                      sm100::smem_desc(b1 + s2 * 2048, 1024, 128), id1, s2 > 0);
#pragma unroll
      for (int s2 = 0; s2 < DK / 16; ++s2)
        sm100::mma_ss(tmem + TM_G + 64, sm100::smem_desc(a2 + s2 * 2048, 1024, 128),
                      sm100::smem_desc(b2 + s2 * 1024, 512, 128), id2, s2 > 0);
      commit_mma();
    }
    wait_mma();
    KDA_PHASE(2);

    // ---- (D) Gram epilogue (warps 0-3) | (beta V)^T (warps 4-7) -------------
    if (warp < 4) {
      const int l = tid;  // TMEM lane
      // diagonal halves: lane l holds row (l & 31) of q0 | k0 | q1 | k1
      {
        const int part = l >> 5, rl = l & 31;
        const int hf = part >> 1, isk = part & 1;
        const int r = 32 * hf + rl, cb = 32 * hf;  // row, first column of the block
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; c += 16) {
          float w16[16];
          sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_G + cb + c), w16);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[c + e] = w16[e];
        }
        sm100::tmem_wait_ld();
        if (!isk) {  // A_qk, inclusive mask; the block above the diagonal is zero
          if (MODE == 0) {
          float t[8];
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
#pragma unroll
            for (int e = 0; e < 8; ++e) t[e] = (cb + 8 * g8 + e <= r) ? v[8 * g8 + e] : 0.0f;
            st8_bf16(smem + OFF_AQ + k64_off(r, cb + 8 * g8), t);
          }
          if (hf == 0) {
            const float z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) st8_bf16(smem + OFF_AQ + k64_off(r, 32 + 8 * g8), z);
          }
          if (dbg && tp.dbg_aqk) {
            for (int c = 0; c < 32; ++c)
              tp.dbg_aqk[(dbo + r) * C + cb + c] = (cb + c <= r) ? v[c] : 0.0f;
            if (hf == 0)
              for (int c = 32; c < C; ++c) tp.dbg_aqk[(dbo + r) * C + c] = 0.0f;
          }
          }
        } else {     // beta_r A_kk, strict mask, fp32 for the solve
          const float br = beta_at(r);
          float4* row = reinterpret_cast<float4*>(s_akk + r * AKK_LD + cb);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            float t4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = 4 * c4 + e;
              t4[e] = (cb + c < r) ? br * v[c] : 0.0f;
            }
            row[c4] = make_float4(t4[0], t4[1], t4[2], t4[3]);
          }
        }
      }
      // cross block (rows 32..63 x columns 0..31) from the M = 64 product:
      // product row m sits in lane 32 * (m / 16) + m % 16
      {
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; c += 16) {
          float w16[16];
          sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_G + 64 + c), w16);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[c + e] = w16[e];
        }
        sm100::tmem_wait_ld();
        if ((l & 31) < 16) {
          const int m = 16 * (l >> 5) + (l & 15);
          const int r = 32 + (m & 31);
          if (m < 32) {  // A_qk[r, 0..31] (the output needs it)
            if (MODE == 0) {
            float t[8];
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
#pragma unroll
              for (int e = 0; e < 8; ++e) t[e] = v[8 * g8 + e];
              st8_bf16(smem + OFF_AQ + k64_off(r, 8 * g8), t);
            }
            if (dbg && tp.dbg_aqk)
              for (int c = 0; c < 32; ++c) tp.dbg_aqk[(dbo + r) * C + c] = v[c];
            }
          } else {       // beta_r A_kk[r, 0..31]
            const float br = beta_at(r);
            float4* row = reinterpret_cast<float4*>(s_akk + r * AKK_LD);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
              row[c4] = make_float4(br * v[4 * c4], br * v[4 * c4 + 1], br * v[4 * c4 + 2],
                                    br * v[4 * c4 + 3]);
          }
        }
      }
    } else {
      const int i = tid - 128;
      // (beta V)^T, K-major [value channel jv][row r]
      const int jv = i & 63, rh = i >> 6;  // rows 32rh .. 32rh+31
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        float t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int r = 32 * rh + 8 * g8 + e;
          t[e] = (r < L) ? beta_at(r) * ld_bf16(smem + OFF_V, sw128_off(r, jv)) : 0.0f;
        }
        st8_bf16(smem + OFF_BV + k64_off(jv, 32 * rh + 8 * g8), t);
      }
    }
    sm100::fence_async_smem();
    sync_all();
    KDA_PHASE(3);

    // ---- (E) T = (I + A_kk)^{-1}, fp32 blocked solve, bf16 T -----------------
    unit_lower_inverse<AKK_LD>(s_akk, s_tf, s_y, smem + OFF_T, tid);
    if (dbg && (tp.dbg_t || tp.dbg_akk)) {
      for (int e = tid; e < C * C; e += kThreads) {
        const int r = e / C, i = e % C;
        if (tp.dbg_t)
          tp.dbg_t[(dbo + r) * C + i] = (i < r) ? s_tf[r * AKK_LD + i] : (i == r ? 1.0f : 0.0f);
        if (tp.dbg_akk)
          tp.dbg_akk[(dbo + r) * C + i] = (i < r) ? s_akk[r * AKK_LD + i] : 0.0f;
      }
    }
    sm100::fence_async_smem();
    sync_all();
    KDA_PHASE(4);

    // ---- (F) W^T and U products --------------------------------------------
    if (tid == 0) {
      const uint32_t idesc = sm100::idesc_bf16(128, 64, 0, 0);
      const uint32_t s_bkg = sm100::smem_u32(smem + OFF_BKG);
      const uint32_t s_t = sm100::smem_u32(smem + OFF_T);
      const uint32_t s_bv = sm100::smem_u32(smem + OFF_BV);
#pragma unroll
      for (int s = 0; s < C / 16; ++s) {
        sm100::mma_ss(tmem + TM_W, sm100::smem_desc(s_bkg + 256 * s, 128, 1024),
                      sm100::smem_desc(s_t + 256 * s, 128, 1024), idesc, s > 0);
      }
#pragma unroll
      for (int s = 0; s < C / 16; ++s) {
        sm100::mma_ss(tmem + TM_U, sm100::smem_desc(s_t + 256 * s, 128, 1024),
                      sm100::smem_desc(s_bv + 256 * s, 128, 1024), idesc, s > 0);
      }
      commit_mma();
    }
    // the landing zone has been read for the last time: prefetch the next chunk
    if (ci + 1 < nchunks) {
      if (tid == 32) issue_tma(ci + 1);
      tma_pending = true;
      tma_parity = (uint32_t)((ci + 1) & 1);
    }
    // while W^T and U are formed: bf16 copy of the entry state S (B of the
    // P product) and S <- gamma_C * S ahead of the rank-64 update (warps
    // 4-7, lane = key channel); neither touches what these products read
    if (warp >= 4) {
      const int i = tid - 128;
      const float gc = s_gc[i];
#pragma unroll 1
      for (int cb = 0; cb < SC; cb += 64) {
        float sv[64];
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          float v[16];
          sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_S + cb + c), v);
#pragma unroll
          for (int e = 0; e < 16; ++e) sv[c + e] = v[e];
        }
        sm100::tmem_wait_ld();
#pragma unroll
        for (int jg = 0; jg < 8; ++jg)
          st8_bf16(smem + OFF_SB + mn_off(cb + 8 * jg, i, SC * 16), sv + 8 * jg);
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          uint32_t r[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(gc * sv[c + e]);
          sm100::tmem_st16(sm100::taddr(tmem, lane_q, TM_S + cb + c), r);
        }
      }
      sm100::tmem_wait_st();
    }
    wait_mma();
    KDA_PHASE(5);

    // ---- (G) W rows into [W; Q gamma] (warps 0-3, lane = key channel) -------
    if (warp < 4) {
      const int j = tid;
      float wv[64];
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        float v[16];
        sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_W + c), v);
#pragma unroll
        for (int e = 0; e < 16; ++e) wv[c + e] = v[e];
      }
      sm100::tmem_wait_ld();
#pragma unroll
      for (int rg = 0; rg < 8; ++rg) st8_bf16(smem + OFF_WQ + mn_off(8 * rg, j, 2048), wv + 8 * rg);
      if (dbg && tp.dbg_w)
        for (int r = 0; r < C; ++r) tp.dbg_w[(dbo + r) * DK + j] = wv[r];
    } else if (dbg_nh && tp.dbg_u && warp < 6) {
      const int r = tid - 128;  // lanes 0..63 of U
      for (int c = 0; c < 64; c += 16) {
        float v[16];
        sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_U + c), v);
        sm100::tmem_wait_ld();
        for (int e = 0; e < 16; ++e) tp.dbg_u[(dbo + r) * DV + half * DVH + c + e] = v[e];
      }
    }
    sm100::fence_async_smem();
    sync_all();
    KDA_PHASE(6);

    // ---- (H) P = [W; Q gamma] . S -------------------------------------------
    if (tid == 0) {
      const uint32_t idesc = sm100::idesc_bf16(128, SC, 1, 1);
      const uint32_t sa = sm100::smem_u32(smem + OFF_WQ);
      const uint32_t sb = sm100::smem_u32(smem + OFF_SB);
#pragma unroll
      for (int s = 0; s < DK / 16; ++s)
        sm100::mma_ss(tmem + TM_P, sm100::smem_desc(sa + s * 4096, 2048, 128),
                      sm100::smem_desc(sb + s * 2 * SC * 16, SC * 16, 128), idesc, s > 0);
      commit_mma();
    }
    // the next chunk's tiles landed during this chunk: its decay factors are
    // computed while the tensor cores work on P
    if (ci + 1 < nchunks) {
      KDA_PHASE(12);
      wait_tma(ci + 1);
      KDA_PHASE(13);
      gate_alpha(ci + 1);
      KDA_PHASE(14);
      // beta of the next chunk, stored at its start
      if (tid < C) {
        const int64_t rn = cs + C + tid;
        beta_next = (rn < t1) ? beta_g[(row_base + rn) * H + h] : (unsigned short)0;
      }
    }
    wait_mma();
    KDA_PHASE(7);

    // ---- (I) Delta = U - W S (warps 0-1, lane = row) ------------------------
    if (warp < 2) {
      const int r = tid;
      float dv[64];
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        float ws[16], u[16];
        sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_P + c), ws);
        sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_U + c), u);
        sm100::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) dv[c + e] = u[e] - ws[e];
      }
#pragma unroll
      for (int jg = 0; jg < 8; ++jg)
        st8_bf16(smem + OFF_DL + mn_off(8 * jg, r, SC * 16), dv + 8 * jg);
      if (MODE == 1) {  // the transition's columns: its "U" is zero
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          float wp[16];
          sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_P + 64 + c), wp);
          sm100::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) dv[c + e] = -wp[e];
        }
#pragma unroll
        for (int jg = 0; jg < 8; ++jg)
          st8_bf16(smem + OFF_DL + mn_off(64 + 8 * jg, r, SC * 16), dv + 8 * jg);
      }
    }
    sm100::fence_async_smem();
    sync_all();
    KDA_PHASE(8);

    // ---- (J) S += (K dec)^T Delta;  O += A_qk Delta ---------------------------
    if (tid == 0) {
      const uint32_t id_s = sm100::idesc_bf16(128, SC, 0, 1);
      const uint32_t s_kd = sm100::smem_u32(smem + OFF_KD);
      const uint32_t s_dl = sm100::smem_u32(smem + OFF_DL);
#pragma unroll
      for (int s = 0; s < C / 16; ++s)
        sm100::mma_ss(tmem + TM_S, sm100::smem_desc(s_kd + 256 * s, 128, 1024),
                      sm100::smem_desc(s_dl + s * 2 * SC * 16, SC * 16, 128), id_s, 1);
      if (MODE == 0) {
        const uint32_t id_o = sm100::idesc_bf16(128, 64, 0, 1);
        const uint32_t s_x = sm100::smem_u32(smem + OFF_X);
#pragma unroll
        for (int s = 0; s < C / 16; ++s)
          sm100::mma_ss(tmem + TM_P, sm100::smem_desc(s_x + 256 * s, 128, 1024),
                        sm100::smem_desc(s_dl + s * 2048, 1024, 128), id_o, 1);
      }
      commit_mma();
    }
    wait_mma();
    KDA_PHASE(9);

    // ---- (K') state checkpoint (warps 4-7, lane = key channel) ------------
    if (MODE == 0 && p.ckpt && warp >= 4 && L == C) {
      const int64_t done = cs + L - t0;
      if (done % p.ckpt_every == 0 && done / p.ckpt_every <= p.ckpt_max) {
        const int i = tid - 128;
        float* dst = p.ckpt + ((((int64_t)n * H + h) * p.ckpt_max + done / p.ckpt_every - 1) *
                                   DK + i) * DV + half * DVH;
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          float v[16];
          sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_S + c), v);
          sm100::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(dst + c + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
      }
    }
    // ---- (K) output rows (warps 2-3, lanes 64..127 = row r) ------------------
    if (MODE == 0 && (warp == 2 || warp == 3)) {
      const int r = tid - 64;
      float o[64];
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        float v[16];
        sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_P + c), v);
#pragma unroll
        for (int e = 0; e < 16; ++e) o[c + e] = v[e];
      }
      sm100::tmem_wait_ld();
      if (r < L) {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) +
                             ((row_base + cs + r) * H + h) * DV + half * DVH;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          uint4 w = make_uint4(sm100::pack_bf16x2(o[8 * g], o[8 * g + 1]),
                               sm100::pack_bf16x2(o[8 * g + 2], o[8 * g + 3]),
                               sm100::pack_bf16x2(o[8 * g + 4], o[8 * g + 5]),
                               sm100::pack_bf16x2(o[8 * g + 6], o[8 * g + 7]));
          *reinterpret_cast<uint4*>(dst + 8 * g) = w;
        }
      }
    }
    const bool aborted_end = sync_aborted(s_abort);
    KDA_PHASE(10);
    if (aborted_end) break;
  }

  // ---- drain anything still in flight after an abort, write the state ----
  // bounded waits for copies and products still in flight before the TMEM
  // is released (only after an abort; otherwise nothing is pending)
  if (*s_abort) {
    if (tma_pending) sm100::mbar_wait(bar_tma, tma_parity, 200000000ull);
    if (mma_inflight) sm100::mbar_wait(bar_mma, mma_phase & 1, 200000000ull);
  }
  // MODE 0: the sequence's final state (from its last segment); MODE 1: the
  // segment's zero-start final state and this half's columns of its
  // cumulative transition into the segment scratch
  if (!*s_abort && warp < 4) {
    const int i = tid;
    float* dst_s = nullptr;
    if (MODE == 0 && sg == nseg - 1 && p.final_state) dst_s = p.final_state + sbase;
    if (MODE == 1) dst_s = p.seg_final + segbase;
    if (dst_s) {
      for (int c = 0; c < DVH; c += 16) {
        float v[16];
        sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_S + c), v);
        sm100::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) dst_s[(int64_t)i * DV + c + e] = v[e];
      }
    }
    if (MODE == 1) {
      float* dst_p = p.seg_P + (((int64_t)n * nseg + sg) * H + h) * (int64_t)DK * DK + half * 64;
      for (int c = 0; c < 64; c += 16) {
        float v[16];
        sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_S + 64 + c), v);
        sm100::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) dst_p[(int64_t)i * DK + c + e] = v[e];
      }
    }
  }
  sm100::tc_fence_before();
  __syncthreads();
  if (warp == 0) sm100::tmem_dealloc(tmem, TM_COLS);
}

// ---------------------------------------------------------------------------

template <int MODE, bool DBG>
kda_status launch_tc(const TcParams& tp, cudaStream_t stream) {
  const kda::FwdParams& p = tp.p;
  const int64_t rows = p.cu_seqlens ? (int64_t)p.T : (int64_t)p.N * p.T;
  const int nseg = p.nseg > 1 ? p.nseg : 1;
  if ((int64_t)p.N * nseg > 65535 || p.H > 65535) return KDA_ERR_UNSUPPORTED;
  if (rows >= (int64_t)1 << 31) return KDA_ERR_UNSUPPORTED;
  CUtensorMap mq, mk, mg, mv;
  if (rows > 0) {
    if (!make_map(&mq, p.q, rows, p.H, DK) || !make_map(&mk, p.k, rows, p.H, DK) ||
        !make_map(&mg, p.g, rows, p.H, DK) || !make_map(&mv, p.v, rows, p.H, DV))
      return KDA_ERR_CUDA;
  } else {
    // an empty batch still passes its states through; the maps are unused
    memset(&mq, 0, sizeof(mq));
    mk = mq; mg = mq; mv = mq;
  }
  if (kda_smem_attr((const void*)kda_tc_fused_kernel<MODE, DBG>, Lay<MODE>::SMEM_BYTES) !=
      KDA_OK)
    return KDA_ERR_CUDA;
  dim3 grid(2, p.H, p.N * nseg);
  kda_tc_fused_kernel<MODE, DBG><<<grid, kThreads, Lay<MODE>::SMEM_BYTES, stream>>>(mq, mk, mg, mv, tp);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

#ifdef KDA_PHASE_TIMING
extern "C" int kda_phase_timing_read(unsigned long long* out16, int reset) {
  if (cudaMemcpyFromSymbol(out16, kda_phase_cycles, sizeof(unsigned long long) * 24) !=
      cudaSuccess)
    return -1;
  if (reset) {
    unsigned long long z[24] = {0};
    cudaMemcpyToSymbol(kda_phase_cycles, z, sizeof(z));
  }
  return 0;
}
#endif

bool kda_tc_supported(int dk, int dv) { return dk == DK && dv == DV; }

kda_status kda_launch_tc(const kda::FwdParams& p, cudaStream_t stream) {
  TcParams tp;
  tp.p = p;
  tp.dbg_n = -1;
  tp.dbg_h = -1;
  tp.dbg_gam = tp.dbg_aqk = tp.dbg_akk = tp.dbg_t = tp.dbg_w = tp.dbg_u = nullptr;
  return launch_tc<0, false>(tp, stream);
}

kda_status kda_launch_tc_summary(const kda::FwdParams& p, cudaStream_t stream) {
  TcParams tp;
  tp.p = p;
  tp.dbg_n = -1;
  tp.dbg_h = -1;
  tp.dbg_gam = tp.dbg_aqk = tp.dbg_akk = tp.dbg_t = tp.dbg_w = tp.dbg_u = nullptr;
  return launch_tc<1, false>(tp, stream);
}

extern "C" kda_status kda_debug_intra(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                      const uint16_t* g_logit, const uint16_t* beta, int B,
                                      int T, int H, int dk, int dv, const int32_t* cu_seqlens,
                                      int n, int h, float* gam, float* aqk, float* akk,
                                      float* tinv, float* w, float* u, kda_stream_t stream) {
  if (!q || !k || !v || !g_logit || !beta) return KDA_ERR_INVALID_ARG;
  if (dk != DK || dv != DV) return KDA_ERR_UNSUPPORTED;
  if (B < 1 || T < 1 || H < 1 || n < 0 || n >= B || h < 0 || h >= H) return KDA_ERR_INVALID_ARG;
  // scratch outputs for the full forward
  const int64_t rows = cu_seqlens ? (int64_t)T : (int64_t)B * T;
  void* out = nullptr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMallocAsync(&out, (size_t)rows * H * DV * 2, s) != cudaSuccess) return KDA_ERR_CUDA;
  TcParams tp;
  tp.p = kda::FwdParams{};
  tp.p.q = q; tp.p.k = k; tp.p.v = v; tp.p.g = g_logit; tp.p.beta = beta;
  tp.p.init_state = nullptr; tp.p.out = out; tp.p.final_state = nullptr;
  tp.p.ckpt = nullptr; tp.p.ckpt_every = 0; tp.p.ckpt_max = 0;
  tp.p.cu_seqlens = cu_seqlens; tp.p.dev_status = nullptr;
  tp.p.N = B; tp.p.T = T; tp.p.H = H; tp.p.dk = dk; tp.p.dv = dv; tp.p.scale = 1.0f;
  tp.dbg_n = n; tp.dbg_h = h;
  // gam is the trigger for the dump; give it a scratch when not wanted
  float* g_scratch = nullptr;
  if (!gam) {
    const int64_t len = cu_seqlens ? (int64_t)T : (int64_t)T;
    if (cudaMallocAsync((void**)&g_scratch, (size_t)(len + C) * DK * 4, s) != cudaSuccess) {
      cudaFreeAsync(out, s);
      return KDA_ERR_CUDA;
    }
  }
  tp.dbg_gam = gam ? gam : g_scratch;
  tp.dbg_aqk = aqk; tp.dbg_akk = akk; tp.dbg_t = tinv; tp.dbg_w = w; tp.dbg_u = u;
  kda_status st = launch_tc<0, true>(tp, s);
  if (g_scratch) cudaFreeAsync(g_scratch, s);
  cudaFreeAsync(out, s);
  return st;
}
