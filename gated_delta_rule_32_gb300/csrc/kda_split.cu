// kda_split.cu -- the two-kernel tensor-core forward (dense and packed batches).
//
// Everything of a chunk that does not depend on the state entering it (the
// gate, the Gram matrices, T = (I + beta A_kk)^{-1}, W = T (beta K gamma),
// U = T (beta V) = (T Diag(beta)) V, Q gamma and K e^{G_C - G}) is
// independent across chunks;
// only Delta = U - W S, O = (Q gamma) S + A_qk Delta and
// S <- gamma_C S + (K dec)^T Delta chain one chunk to the next (Towards AI
// walkthrough, "Infrastructure co-design": the chunk-to-chunk state
// dependency is the only serial part).  So:
//   intra kernel  persistent, two CTAs per SM walking the (sequence, head,
//                 chunk) items; writes one record per chunk to global
//                 memory, laid out as the state kernel's shared-memory image;
//   state kernel  one CTA per (half of the value channels, head, sequence);
//                 per chunk a bulk copy of the record and a TMA load of its
//                 half of V straight from the input, the U product of its
//                 half (off the chain: it runs while the CUDA cores copy the
//                 state), then two tensor-core products and two short
//                 epilogues on the chain, the state in tensor memory
//                 throughout.
// The record holds bf16 operands (W, Q gamma, K dec, A_qk, T Diag(beta)) and
// fp32 gamma_C; U is accumulated in fp32 from the bf16 T Diag(beta) and the
// input's own bf16 V, so V is never rewritten and the record carries nothing
// of the size of V.
//
// A long sequence runs in slices of chunks (intra kernel over the slice,
// then the state kernel over it), so the record buffer stays bounded; the
// state crosses slice boundaries through global memory.  Packed batches
// (cu_seqlens) run in slices of chunk columns.  A dense batch of few long
// sequences is cut into segments whose chains run side by side, joined by
// the affine composition of each segment's zero-start state and cumulative
// transition (orkas.ai, "Kimi K3 architecture", "The cost is paid in the
// serving stack": the context-parallel decomposition, here across the SMs
// of one GPU).
#include <cudaTypedefs.h>
#include <string.h>

#include <atomic>
#include <map>
#include <mutex>

#include "kda_common.cuh"
#include "sm100.cuh"
#include "kda_tc_util.cuh"

namespace {

using namespace kda_tc;

constexpr int DK = 128, DV = 128, C = 64;
constexpr int kThreads = 256;
constexpr int AKK_LD = 72;

// ---- chunk record (bytes) ---------------------------------------------------
constexpr int REC_KD = 0;        // (K dec)^T, K-major [key channel j][row r]  16384
constexpr int REC_AQ = 16384;    // A_qk masked (i <= r), K-major [r][i]         8192
constexpr int REC_WQ = 24576;    // [W; Q gamma], MN-major 128 rows x 128 K     32768
constexpr int REC_T = 57344;     // T Diag(beta), K-major [r][i]                  8192
constexpr int REC_GC = 65536;    // gamma_C fp32 [128]                             512
constexpr int REC_BYTES = 66048;
// what one state CTA holds per chunk: the record (KD | AQ | WQ | T Diag(beta)
// by one bulk copy, gamma_C by another) and the 64 value channels of its half
// of V, loaded from the input by one TMA box of 64 rows x 128 bytes with the
// 128-byte swizzle: an MN-major operand (N = value channel, K = row) in
// swizzle atoms of 8 rows, 1024 bytes apart.  U = T Diag(beta) V of the half
// is formed there, on the tensor cores, into tensor memory: its rows past 63
// read the V tile that follows T and are never used.  Stages are a multiple
// of 1024 bytes, so the V tile stays aligned to its atoms.
constexpr int ST_KD = 0, ST_AQ = 16384, ST_WQ = 24576, ST_T = 57344, ST_V = 65536,
              ST_GC = 73728;
constexpr int STAGE_BYTES = 74752;
static_assert(STAGE_BYTES % 1024 == 0 && ST_V % 1024 == 0, "swizzle atoms of V");
static_assert(ST_GC + 512 <= STAGE_BYTES, "stage");
constexpr int ST_COPY = REC_GC;  // bytes of the record's first bulk copy
static_assert(ST_V == ST_T + 8192, "U operand rows");
static_assert(ST_COPY == ST_V, "first bulk copy ends where V starts");

struct SplitParams {
  kda::FwdParams p;
  unsigned char* rec;  // records: dense [N][H][c_count], packed [H][g_count]
  int c_begin;         // first chunk of the slice (dense)
  int c_count;         // chunks in the slice (dense)
  const float* s_in;   // state entering the slice [N][H][DK][DV] (null: zero)
  float* s_out;        // state leaving the slice (null: not kept)
  // packed batches (cu_seqlens): sequence n owns the chunk columns
  // [chunk_off[n], chunk_off[n + 1]); column g starts at token row
  // chunk_tab[g].x and holds chunk_tab[g].y >> 24 rows (0: no chunk); a
  // slice is the columns [g_begin, g_begin + g_count)
  const int2* chunk_tab;  // [g_max], null for dense batches
  const int* chunk_off;   // [N + 1]
  // the sequence each state CTA z runs (longest first), [N]; null: z itself
  const int* seq_order;
  int g_max;              // chunk columns: ceil(T / 64) + N bounds the true count
  int g_begin, g_count;
  // extents the debug build checks accesses against: chunk records the
  // workspace holds, token rows of the input tensors
  int64_t rec_items;
  int64_t rows;
  // test hook (0 in every normal call): bit 0 makes the intra kernel's first
  // wait, bit 1 the state kernel's first wait, wait on a barrier that nothing
  // ever completes, with a 1 ms limit, so that the timeout and abort path runs
  int stall_test;
  // segments of a dense batch (seg_g > 1; records of every chunk at hand):
  // sequence n is cut into seg_g segments of seg_len chunks (the last one
  // shorter), state grid z = n * seg_g + segment.  seg_pass 1: segment 0 in
  // full (from init_state, its final state into seg_entry[n][1]); segments
  // 1 .. seg_g - 2 from a zero state (final into seg_s0) and their
  // cumulative transitions (grid x = 2, 3: the state run from the identity
  // with U = 0, final into seg_trans).  seg_pass 2: segments 1 .. seg_g - 1
  // in full from seg_entry (the last one's final state into final_state).
  // Buffers [N][seg_g][H][DK][DV] (seg_trans: [DK][DK]).
  int seg_g, seg_len, seg_pass;
  // dense records laid out for every chunk of a sequence (record of chunk c
  // at (n * H + h) * rec_stride + c) instead of for the slice; 0: the slice
  int rec_stride;
  float* seg_entry;
  float* seg_s0;
  float* seg_trans;
};

// limit of the waits the stall test makes run out
constexpr unsigned long long kStallTestNs = 1000000ull;

#ifdef KDA_PHASE_TIMING
// cycles per phase, summed over the CTAs of (sequence 0, head 0) for the
// intra kernel (marks 0..11) and over chunks of one state CTA (16..23);
// instrumented builds only
__device__ unsigned long long kda_split_cycles[32];
#define SPLIT_MARK(k, cond)                                                    \
  do {                                                                         \
    if (cond) {                                                                \
      const long long t_ = clock64();                                          \
      atomicAdd(&kda_split_cycles[k], (unsigned long long)(t_ - t_mark));      \
      t_mark = t_;                                                             \
    }                                                                          \
  } while (0)
#else
#define SPLIT_MARK(k, cond) do { } while (0)
#endif

__device__ __forceinline__ void record_error(const kda::FwdParams& p, int* s_abort,
                                             kda_status st) {
  *s_abort = 1;
  if (p.dev_status) atomicExch(p.dev_status, (int32_t)st);
}

// ===========================================================================
// intra kernel
// ===========================================================================
// shared memory (bytes); 110 KiB so that two CTAs share an SM
constexpr int I_Q = 0, I_K = 16384, I_G = 32768;  // TMA landing, 2 unswizzled boxes of 64 channels
constexpr int I_OB = 49152;                        // Gram operands for 64 key channels
constexpr int I_A1 = I_OB;                         // [q0; k0; q1; k1] MN-major 128 x 64
constexpr int I_B1 = I_OB + 16384;                 // [c0; c1]          MN-major  64 x 64
constexpr int I_A2 = I_OB + 24576;                 // [q1'; k1']        MN-major  64 x 64
constexpr int I_B2 = I_OB + 32768;                 // c0'               MN-major  32 x 64
constexpr int I_KG = I_OB + 36864;                 // (K gamma)^T K-major 128 x 64
constexpr int I_BETA = I_KG + 16384;               // 64 raw bf16
constexpr int I_PT = I_BETA + 128;                 // [4 tiles][128] fp32 tile products
static_assert(I_BETA % 16 == 0, "beta rows are read 8 at a time");
constexpr int I_BAR = I_PT + 2048;
constexpr int I_MISC = I_BAR + 64;
constexpr int I_T = I_MISC + 64;                   // T bf16 K-major [r][i] (8192)
constexpr int I_SMEM = I_T + 8192;
static_assert(I_T % 16 == 0, "T is an operand and a bulk-copy source");
// the solve's scratch overlays what is dead by then
constexpr int I_AKK = I_OB, I_TF = I_OB + 18432;   // [64][72] fp32 each (after the Grams)
constexpr int I_Y = I_Q + 8192;                    // Y fp32 [32][36] (the solve, over dead Q)
static_assert(I_TF + 64 * AKK_LD * 4 <= I_KG, "solve scratch");
static_assert(I_Y + 32 * 36 * 4 <= I_K, "block-merge scratch");
static_assert(2 * (I_SMEM + 1024) <= 233472, "two CTAs per SM");
constexpr uint32_t I_TM_COLS = 256;
constexpr uint32_t TM_G = 0;     // Gram products: [0, 64) diagonal halves, [64, 96) cross
constexpr uint32_t TM_W = 128;   // W^T, read out while the next item's Grams are formed

__global__ void __launch_bounds__(kThreads, 2)
    kda_tc_intra_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_g, const SplitParams sp) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const kda::FwdParams& p = sp.p;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = p.H;
  // work items: dense w = (n * H + h) * c_count + chunk of the slice,
  // packed w = chunk column of the slice * H + h; this CTA takes blockIdx.x,
  // blockIdx.x + gridDim.x, ...
  const bool packed = sp.chunk_tab != nullptr;
  const int64_t n_items = packed ? (int64_t)sp.g_count * H : (int64_t)p.N * H * sp.c_count;
  struct Item {
    int n, h, cl;    // sequence, head, chunk of the slice (packed: column of the slice)
    int L;           // valid rows of the chunk
    int64_t row0;    // global row of its first token
    int64_t w;
    int64_t ri;      // its record
  };
  auto finish = [&](Item& it) {
    if (packed) {  // (read well before its first use, the next item's tiles)
      const int2 e = it.w < n_items ? sp.chunk_tab[sp.g_begin + it.cl] : make_int2(0, 0);
      it.row0 = e.x;
      it.n = e.y & 0xFFFFFF;
      it.L = (e.y >> 24) & 0x7F;
      it.ri = (int64_t)it.h * sp.g_count + it.cl;
    } else {
      const int64_t cs = ((int64_t)sp.c_begin + it.cl) * C;
      it.L = (p.T - cs) < C ? (int)(p.T - cs) : C;
      it.row0 = (int64_t)it.n * p.T + cs;
      it.ri = sp.rec_stride > 0
                  ? ((int64_t)it.n * H + it.h) * sp.rec_stride + sp.c_begin + it.cl
                  : it.w;
    }
  };
  // the coordinates of item w (divisions: once per CTA), and those of the
  // item gridDim.x further on, by carries (32-bit adds only)
  auto item_of = [&](int64_t w) {
    Item it;
    if (packed) {
      it.h = (int)(w % H);
      it.cl = (int)(w / H);
      it.n = 0;
    } else {
      const int nh = (int)(w / sp.c_count);
      it.cl = (int)(w % sp.c_count);
      it.h = nh % H;
      it.n = nh / H;
    }
    it.w = w;
    finish(it);
    return it;
  };
  const int step_cl = packed ? (int)(gridDim.x / H) : (int)(gridDim.x % sp.c_count);
  const int step_nh = packed ? 0 : (int)(gridDim.x / sp.c_count);
  const int step_h = packed ? (int)(gridDim.x % H) : step_nh % H, step_n = step_nh / H;
  auto next_of = [&](const Item& a) {
    Item it;
    it.w = a.w + gridDim.x;
    if (packed) {
      it.h = a.h + step_h;
      const int carry = it.h >= H;
      if (carry) it.h -= H;
      it.cl = a.cl + step_cl + carry;
      it.n = 0;
    } else {
      it.cl = a.cl + step_cl;
      const int carry = it.cl >= sp.c_count;
      if (carry) it.cl -= sp.c_count;
      it.h = a.h + step_h + carry;
      it.n = a.n + step_n;
      if (it.h >= H) {
        it.h -= H;
        it.n += 1;
      }
    }
    finish(it);
    return it;
  };
#ifdef KDA_PHASE_TIMING
  long long t_mark = clock64();
  const bool mk = tid == 0 && blockIdx.x == 0;
#endif

  uint64_t* bar_q = reinterpret_cast<uint64_t*>(smem + I_BAR);  // Q tiles
  uint64_t* bar_g = bar_q + 1;                                   // decay-logit tiles
  uint64_t* bar_k = bar_q + 2;                                   // K tiles
  uint64_t* bar_mma = bar_q + 3;
  uint64_t* bar_never = bar_q + 4;  // stall test only: nothing arrives on it
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + I_MISC);
  int* s_abort = reinterpret_cast<int*>(smem + I_MISC + 4);
  unsigned short* s_beta_raw = reinterpret_cast<unsigned short*>(smem + I_BETA);
  auto beta_at = [&](int r) { return __uint_as_float((uint32_t)s_beta_raw[r] << 16); };
  float* s_pt = reinterpret_cast<float*>(smem + I_PT);

  if (warp == 0) {
    sm100::tmem_alloc(s_tmem, I_TM_COLS);
    sm100::tmem_relinquish();
  }
  // the tiles of an item land region by region as the previous item's use
  // of that region ends (issued by thread 32)
  auto load_q = [&](const Item& it) {
    sm100::mbar_arrive_expect_tx(bar_q, 16384);
    sm100::tma_load_3d(smem + I_Q, &tm_q, bar_q, 0, it.h, (int)it.row0);
    sm100::tma_load_3d(smem + I_Q + 8192, &tm_q, bar_q, 64, it.h, (int)it.row0);
  };
  auto load_g = [&](const Item& it) {
    sm100::mbar_arrive_expect_tx(bar_g, 16384);
    sm100::tma_load_3d(smem + I_G, &tm_g, bar_g, 0, it.h, (int)it.row0);
    sm100::tma_load_3d(smem + I_G + 8192, &tm_g, bar_g, 64, it.h, (int)it.row0);
  };
  auto load_k = [&](const Item& it) {
    sm100::mbar_arrive_expect_tx(bar_k, 16384);
    sm100::tma_load_3d(smem + I_K, &tm_k, bar_k, 0, it.h, (int)it.row0);
    sm100::tma_load_3d(smem + I_K + 8192, &tm_k, bar_k, 64, it.h, (int)it.row0);
  };
  // beta of an item, kept as raw bf16 bits in a register until its slot is free
  auto load_beta = [&](const Item& it) -> unsigned short {
    if (tid < C && tid < it.L) {
      if (kda::kDebugChecks && (it.row0 + tid < 0 || it.row0 + tid >= sp.rows)) return 0;
      return static_cast<const unsigned short*>(p.beta)[(it.row0 + tid) * H + it.h];
    }
    return 0;
  };
  Item cur = item_of(blockIdx.x);
  if (tid == 32) {
    sm100::mbar_init(bar_q, 1);
    sm100::mbar_init(bar_g, 1);
    sm100::mbar_init(bar_k, 1);
    sm100::mbar_init(bar_mma, 1);
    sm100::mbar_init(bar_never, 1);
    sm100::fence_mbar_init();
    if (cur.w < n_items) {
      load_g(cur);
      load_q(cur);
      load_k(cur);
    }
  }
  unsigned short beta_raw = cur.w < n_items ? load_beta(cur) : (unsigned short)0;
  if (tid == 0) *s_abort = 0;
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_q = 32u * (warp & 3);  // this warp's TMEM lane quarter
  SPLIT_MARK(0, mk);

  bool mma_pending = false;
  uint32_t mma_phase = 0;
  // items whose copies were issued / waited for, per barrier
  const int first = cur.w < n_items ? 1 : 0;
  int q_issued = first, g_issued = first, k_issued = first;
  int q_done = 0, g_done = 0, k_done = 0;
  auto wait_mma = [&]() {
    const bool ok = sm100::mbar_wait(bar_mma, mma_phase & 1);
    if (ok) ++mma_phase;
    else record_error(p, s_abort, KDA_ERR_TIMEOUT);
    mma_pending = !ok;
    sm100::tc_fence_after();
  };
  auto sync_all = [&]() {
    sm100::tc_fence_before();
    __syncthreads();
    sm100::tc_fence_after();
  };

  // W rows of an item into its record (all warps: lane = key channel, 32
  // rows each), from tensor memory
  auto w_out = [&](unsigned char* r) {
    const int j = tid & 127, rb = (warp >> 2) * 32;
    float wv[32];
#pragma unroll
    for (int c = 0; c < 32; c += 16) {
      float v[16];
      sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_W + rb + c), v);
#pragma unroll
      for (int e = 0; e < 16; ++e) wv[c + e] = v[e];
    }
    sm100::tmem_wait_ld();
#pragma unroll
    for (int rg = 0; rg < 4; ++rg)
      st8_bf16(r + REC_WQ + mn_off(rb + 8 * rg, j, 2048), wv + 8 * rg);
  };
  unsigned char* w_rec = nullptr;  // item whose W product is in flight

  for (int li = 0; cur.w < n_items; ++li) {
    const int L = cur.L;
    unsigned char* rec = sp.rec + cur.ri * (int64_t)REC_BYTES;
    // debug build: the item's record and rows inside their buffers, else the
    // loop ends at the first barrier below, before any global store
    if (kda::kDebugChecks &&
        (cur.ri < 0 || cur.ri >= sp.rec_items || cur.row0 < 0 || cur.row0 + L > sp.rows))
      record_error(p, s_abort, KDA_ERR_BOUNDS);
    const Item nxt = next_of(cur);
    const bool has_next = nxt.w < n_items;
    const uint32_t par = (uint32_t)(li & 1);
    const bool stall = (sp.stall_test & 1) && li == 0;
    if (!(stall ? sm100::mbar_wait(bar_never, 0, kStallTestNs) : sm100::mbar_wait(bar_g, par)))
      record_error(p, s_abort, KDA_ERR_TIMEOUT);
    else g_done = li + 1;
    if (tid < C) s_beta_raw[tid] = beta_raw;  // bf16 bits; readers widen them
    // rows past the end of the sequence (its last chunk only): a decay logit
    // far below zero (alpha = 1), so that no later step masks
    if (L < C) {
      for (int e = tid; e < (C - L) * 16; e += kThreads) {
        const int r = L + (e >> 4), box = (e >> 3) & 1, piece = e & 7;
        const uint32_t ng = 0xC61CC61Cu;  // bf16 pair (-9984, -9984)
        *reinterpret_cast<uint4*>(smem + I_G + box * 8192 + r * 128 + piece * 16) =
            make_uint4(ng, ng, ng, ng);
      }
      __syncthreads();
    }
    SPLIT_MARK(1, mk);

    // ---- gate, pass 0: decay factors of 16 rows (tile a) of key channels
    //      jl and 64 + jl, and the tile products -------------------------------
    const int jl = tid & 63, a = tid >> 6;
    float al0[16], al1[16];
    {
      const unsigned char* g0 = smem + I_G;
      const unsigned char* g1 = smem + I_G + 8192;
      float p0 = 1.0f, p1 = 1.0f;
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        const int r = 16 * a + s;
        const uint32_t o = row_off(r, jl);
        al0[s] = alpha_of(ld_bf16(g0, o));
        al1[s] = alpha_of(ld_bf16(g1, o));
        p0 *= al0[s];
        p1 *= al1[s];
      }
      s_pt[a * 128 + jl] = p0;
      s_pt[a * 128 + 64 + jl] = p1;
    }
    sm100::fence_async_smem();
    if (sync_aborted(s_abort)) break;
    // the decay logits live on in registers only: the next item's G tiles,
    // and its beta (an item ahead of its use)
    if (has_next) {
      if (tid == 32) load_g(nxt);
      g_issued = li + 2;
      beta_raw = load_beta(nxt);
    }
    // the previous item's W product (its rows go out during this item's
    // first Gram product); its T copy has left shared memory before this
    // item's solve rewrites it (a thread that saw the wait fail skips the
    // rows; the loop leaves at the next check that follows a barrier)
    if (w_rec) {
      wait_mma();
      if (tid == 32) sm100::bulk_wait_read();
    }
    SPLIT_MARK(2, mk);

    // ---- gate, pass hk: key channels 64 hk .. 64 hk + 63 -------------------
    // Row/column factors of the two-level Gram scheme (reference points: end
    // of tile 0 for the first half, end of tile 2 for the second, end of
    // tile 1 for the cross block), each a within-tile product E (prefix,
    // row included) or F (suffix, row excluded) times a per-tile constant:
    //   half 0: row e^{G_r - G_15}, col e^{G_15 - G_i}, cross col e^{G_31 - G_i}
    //   half 1: row e^{G_r - G_47}, col e^{G_47 - G_i}, cross row e^{G_r - G_31}
    // and the record's operands Q gamma (e^{G_r}), K dec (e^{G_C - G_r}),
    // with (K gamma)^T kept for the W product (beta enters W through T).
    auto gate_pass = [&](const float (&al)[16], const int hk) {
      const int j = 64 * hk + jl;
      const unsigned char* sq = smem + I_Q + hk * 8192;
      const unsigned char* sk = smem + I_K + hk * 8192;
      const float P0 = s_pt[j], P1 = s_pt[128 + j], P2 = s_pt[256 + j], P3 = s_pt[384 + j];
      if (a == 0) reinterpret_cast<float*>(rec + REC_GC)[j] = P0 * P1 * P2 * P3;
      const int pr = a >> 1, tt = a & 1;
      // tile products are >= e^-80, so their inverses stay below e^80
      const float invPa = __fdividef(1.0f, pr == 0 ? P0 : P2);
      const float invPb = __fdividef(1.0f, pr == 0 ? P1 : P3);
      const float pre = a == 0 ? 1.0f : a == 1 ? P0 : a == 2 ? P0 * P1 : P0 * P1 * P2;
      const float post = a == 0 ? P1 * P2 * P3 : a == 1 ? P2 * P3 : a == 2 ? P3 : 1.0f;
      const float rs = tt == 0 ? invPa : 1.0f;   // diagonal-half row factor
      const float cf = tt == 0 ? 1.0f : invPb;   // diagonal-half column factor
      // cross-block factor: column (first half) or row (second half)
      const float xf = pr == 0 ? (tt == 0 ? P1 : 1.0f) : (tt == 0 ? 1.0f : P2);
      // q's factors carry the scale
      const float rsq = rs * p.scale, xfq = xf * p.scale, preq = pre * p.scale;
      float F[16];
      {
        float f = 1.0f;
#pragma unroll
        for (int s = 15; s >= 0; --s) { F[s] = f; f *= al[s]; }
      }
      float e = 1.0f;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int r0 = 16 * a + 8 * g;  // chunk row of this group of 8
        float qE[8], kE[8], kF[8], t[8];
#pragma unroll
        for (int e8 = 0; e8 < 8; ++e8) {
          const int r = r0 + e8;
          const uint32_t o = row_off(r, jl);
          const float qv = ld_bf16(sq, o);
          const float kv = ld_bf16(sk, o);
          e *= al[8 * g + e8];
          qE[e8] = qv * e;
          kE[e8] = kv * e;
          kF[e8] = kv * F[8 * g + e8];
        }
        if (pr == 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = qE[i] * rsq;
          st8_bf16(smem + I_A1 + mn_off(r0, jl, 2048), t);
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = kE[i] * rs;
          st8_bf16(smem + I_A1 + mn_off(32 + r0, jl, 2048), t);
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = kF[i] * cf;
          st8_bf16(smem + I_B1 + mn_off(r0, jl, 1024), t);
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = kF[i] * xf;
          st8_bf16(smem + I_B2 + mn_off(r0, jl, 512), t);
        } else {
          const int rr0 = r0 - 32;
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = qE[i] * rsq;
          st8_bf16(smem + I_A1 + mn_off(64 + rr0, jl, 2048), t);
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = kE[i] * rs;
          st8_bf16(smem + I_A1 + mn_off(96 + rr0, jl, 2048), t);
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = qE[i] * xfq;
          st8_bf16(smem + I_A2 + mn_off(rr0, jl, 1024), t);
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = kE[i] * xf;
          st8_bf16(smem + I_A2 + mn_off(32 + rr0, jl, 1024), t);
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = kF[i] * cf;
          st8_bf16(smem + I_B1 + mn_off(32 + rr0, jl, 1024), t);
        }
        // Q gamma into rows 64.. of the record's [W; Q gamma]
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = qE[i] * preq;
        st8_bf16(rec + REC_WQ + mn_off(64 + r0, j, 2048), t);
        // (K gamma)^T, K-major [j][r]
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = kE[i] * pre;
        st8_bf16(smem + I_KG + k64_off(j, r0), t);
        // (K e^{G_C - G})^T, K-major [j][r]
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = kF[i] * post;
        st8_bf16(rec + REC_KD + k64_off(j, r0), t);
      }
    };
    // Gram products over the 64 key channels of one pass: diagonal halves
    // (M = 128, N = 64) and the cross block (M = 64, N = 32)
    auto gram_mma = [&](const int hk) {
      if (tid == 0) {
        const uint32_t id1 = sm100::idesc_bf16(128, 64, 1, 1);
        const uint32_t id2 = sm100::idesc_bf16(64, 32, 1, 1);
        const uint32_t a1 = sm100::smem_u32(smem + I_A1), b1 = sm100::smem_u32(smem + I_B1);
        const uint32_t a2 = sm100::smem_u32(smem + I_A2), b2 = sm100::smem_u32(smem + I_B2);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          sm100::mma_ss(tmem + TM_G, sm100::smem_desc(a1 + s * 4096, 2048, 128),
                        sm100::smem_desc(b1 + s * 2048, 1024, 128), id1, (hk | s) > 0);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          sm100::mma_ss(tmem + TM_G + 64, sm100::smem_desc(a2 + s * 2048, 1024, 128),
                        sm100::smem_desc(b2 + s * 1024, 512, 128), id2, (hk | s) > 0);
        sm100::mma_commit(bar_mma);
      }
      mma_pending = true;
    };

    if (!sm100::mbar_wait(bar_q, par)) record_error(p, s_abort, KDA_ERR_TIMEOUT);
    else q_done = li + 1;
    if (!sm100::mbar_wait(bar_k, par)) record_error(p, s_abort, KDA_ERR_TIMEOUT);
    else k_done = li + 1;
    if (L < C) {  // q = k = 0 past the end of the sequence
      for (int e = tid; e < (C - L) * 16; e += kThreads) {
        const int r = L + (e >> 4), box = (e >> 3) & 1, piece = e & 7;
        const uint32_t off = box * 8192 + r * 128 + piece * 16;
        *reinterpret_cast<uint4*>(smem + I_Q + off) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(smem + I_K + off) = make_uint4(0, 0, 0, 0);
      }
      __syncthreads();
    }
    gate_pass(al0, 0);
    sm100::fence_async_smem();
    sync_all();
    SPLIT_MARK(3, mk);
    gram_mma(0);
    // the previous item's W rows, while the tensor cores form the Grams
    // (W has its own tensor-memory columns)
    if (w_rec) {
      if (!*s_abort) w_out(w_rec);
      w_rec = nullptr;
    }
    wait_mma();
    SPLIT_MARK(4, mk);
    gate_pass(al1, 1);
    sm100::fence_async_smem();
    if (sync_aborted(s_abort)) break;
    SPLIT_MARK(5, mk);
    // K has been read for the last time: the next item's K tiles
    if (has_next) {
      if (tid == 32) load_k(nxt);
      k_issued = li + 2;
    }
    gram_mma(1);
    wait_mma();
    SPLIT_MARK(6, mk);

    // ---- Gram epilogue: diagonal halves (warps 0-3) | cross block (warps 4-7)
    float* s_akk = reinterpret_cast<float*>(smem + I_AKK);
    const int l = tid & 127;  // TMEM lane
    if (warp < 4) {
      {  // diagonal halves: lane l holds row (l & 31) of q0 | k0 | q1 | k1
        const int part = l >> 5, rl = l & 31;
        const int hf = part >> 1, isk = part & 1;
        const int r = 32 * hf + rl, cb = 32 * hf;
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; c += 16) {
          float w16[16];
          sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_G + cb + c), w16);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[c + e] = w16[e];
        }
        sm100::tmem_wait_ld();
        if (!isk) {  // A_qk, inclusive mask; the block right of the diagonal is zero
          float t[8];
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
#pragma unroll
            for (int e = 0; e < 8; ++e) t[e] = (cb + 8 * g8 + e <= r) ? v[8 * g8 + e] : 0.0f;
            st8_bf16(rec + REC_AQ + k64_off(r, cb + 8 * g8), t);
          }
          if (hf == 0) {
            const float z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) st8_bf16(rec + REC_AQ + k64_off(r, 32 + 8 * g8), z);
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
    } else {
      {  // cross block (rows 32..63 x columns 0..31): product row m in lane
         // 32 (m / 16) + m % 16
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
          if (m < 32) {  // A_qk[r, 0..31]
            float t[8];
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
#pragma unroll
              for (int e = 0; e < 8; ++e) t[e] = v[8 * g8 + e];
              st8_bf16(rec + REC_AQ + k64_off(r, 8 * g8), t);
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
    }
    sm100::fence_async_smem();
    if (sync_aborted(s_abort)) break;
    SPLIT_MARK(7, mk);

    // ---- T = (I + beta A_kk)^{-1}, written as T Diag(beta) ------------------
    unit_lower_inverse<AKK_LD>(s_akk, reinterpret_cast<float*>(smem + I_TF),
                               reinterpret_cast<float*>(smem + I_Y), smem + I_T, tid,
                               [&](int i) { return beta_at(i); });
    sm100::fence_async_smem();
    sync_all();
    SPLIT_MARK(8, mk);
    // T Diag(beta) into the record by one bulk copy; the solve scratch (over
    // Q's landing zone) is dead: the next item's Q tiles
    if (tid == 32) {
      sm100::bulk_store(rec + REC_T, smem + I_T, 8192);
      sm100::bulk_commit();
    }
    if (has_next) {
      if (tid == 32) load_q(nxt);
      q_issued = li + 2;
    }

    // ---- W^T = (K gamma)^T (T Diag(beta))^T (U = T Diag(beta) V is formed
    //      by the state kernel from the record's T Diag(beta) and the input V)
    if (tid == 0) {
      const uint32_t idw = sm100::idesc_bf16(128, 64, 0, 0);
      const uint32_t s_kg = sm100::smem_u32(smem + I_KG);
      const uint32_t s_t = sm100::smem_u32(smem + I_T);
#pragma unroll
      for (int s = 0; s < C / 16; ++s)
        sm100::mma_ss(tmem + TM_W, sm100::smem_desc(s_kg + 256 * s, 128, 1024),
                      sm100::smem_desc(s_t + 256 * s, 128, 1024), idw, s > 0);
      sm100::mma_commit(bar_mma);
    }
    // the product is waited for (and W read out) after the next item's
    // decay map, which it overlaps
    mma_pending = true;
    w_rec = rec;
    SPLIT_MARK(9, mk);
    SPLIT_MARK(10, mk);
#ifdef KDA_PHASE_TIMING
    if (mk) atomicAdd(&kda_split_cycles[12], 1ull);  // items measured
#endif
    cur = nxt;
  }

  // the last item's W product
  if (!*s_abort && w_rec) {
    wait_mma();
    if (!*s_abort) w_out(w_rec);
  }
  // after an abort: bounded waits for copies and products still in flight
  // before the shared and tensor memory are released (at most one copy per
  // barrier is outstanding)
  if (*s_abort) {
    if (q_issued > q_done) sm100::mbar_wait(bar_q, q_done & 1, 200000000ull);
    if (g_issued > g_done) sm100::mbar_wait(bar_g, g_done & 1, 200000000ull);
    if (k_issued > k_done) sm100::mbar_wait(bar_k, k_done & 1, 200000000ull);
    if (mma_pending) sm100::mbar_wait(bar_mma, mma_phase & 1, 200000000ull);
  }
  if (tid == 32) sm100::bulk_wait();  // the last T copy
  sm100::tc_fence_before();
  __syncthreads();
  if (warp == 0) sm100::tmem_dealloc(tmem, I_TM_COLS);
  SPLIT_MARK(11, mk);
}

// ===========================================================================
// state kernel
// ===========================================================================
constexpr int S_SB = 2 * STAGE_BYTES;  // S bf16, MN-major (K = key channel) 128 x 64
constexpr int S_DL = S_SB + 16384;     // Delta bf16, MN-major (K = row) 64 x 64
constexpr int S_BAR = S_DL + 8192;
constexpr int S_MISC = S_BAR + 64;
constexpr int S_SMEM = S_MISC + 64;
static_assert(S_SMEM <= 232448, "shared memory");
constexpr uint32_t S_TM_COLS = 256;
constexpr uint32_t TM_S = 0;    // state half: 128 lanes (key channel) x 64 columns
constexpr uint32_t TM_P = 64;   // two buffers of [W S; Q gamma S (+ A_qk Delta)], 64 columns each
constexpr uint32_t TM_U = 192;  // U = T Diag(beta) V of the half (lanes 0..63 = rows)

__global__ void __launch_bounds__(kThreads, 1)
    kda_tc_state_kernel(const __grid_constant__ CUtensorMap tm_v, const SplitParams sp) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const kda::FwdParams& p = sp.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg_g = sp.seg_g > 1 ? sp.seg_g : 1;
  const int half = blockIdx.x & 1, h = blockIdx.y, H = p.H;
  const int n = sp.seq_order ? sp.seq_order[blockIdx.z] : (int)blockIdx.z;
  // segments: pass 1 grid x = [segment 0: 2 halves][segments 1 .. G - 2:
  // (state run, transition run) x 2 halves], pass 2 grid x = [segments
  // 1 .. G - 1: 2 halves].  A transition run starts from the identity, with
  // U = 0 and no output.
  int seg = 0;
  bool trans = false;
  if (seg_g > 1) {
    if (sp.seg_pass == 1) {
      if (blockIdx.x >= 2) {
        seg = 1 + (int)((blockIdx.x - 2) >> 2);
        trans = (((blockIdx.x - 2) >> 1) & 1) != 0;
      }
    } else {
      seg = 1 + (int)(blockIdx.x >> 1);
    }
  }
#ifdef KDA_PHASE_TIMING
  long long t_mark = clock64();
  const bool mk = tid == 0 && half == 0 && h == 0 && n == 0;
#endif
  // this sequence: its chunks of the slice (the first one is chunk c_first
  // of the sequence), their records, its first token row and length, and
  // where its state enters and leaves the slice
  int nc, c_first;
  int64_t row_base, seq_len;
  const unsigned char* rec0;
  const float* s_in = sp.s_in;
  float* s_out = sp.s_out;
  bool involved = true;  // false: the sequence has nothing in this slice
  bool emit = true;      // output rows written
  int64_t in_base = ((int64_t)n * H + h) * (int64_t)DK * DV + half * 64;
  int64_t out_base = in_base;
  if (sp.chunk_tab) {
    const int c_lo = sp.chunk_off[n], c_hi = sp.chunk_off[n + 1];
    const int g0 = sp.g_begin, g1 = sp.g_begin + sp.g_count;
    const int lo = c_lo > g0 ? c_lo : g0, hi = c_hi < g1 ? c_hi : g1;
    nc = hi > lo ? hi - lo : 0;
    c_first = lo - c_lo;
    row_base = p.cu_seqlens[n];
    seq_len = p.cu_seqlens[n + 1] - row_base;
    rec0 = sp.rec + ((int64_t)h * sp.g_count + (lo - g0)) * REC_BYTES;
    // an empty sequence belongs to the slice its (empty) column range starts in
    involved = nc > 0 || (c_lo == c_hi && c_lo >= g0 && c_lo < g1);
    s_in = c_lo >= g0 ? p.init_state : sp.s_in;      // starts here, or carried in
    s_out = c_hi <= g1 ? p.final_state : sp.s_out;   // ends here, or carried on
  } else {
    nc = sp.c_count;
    c_first = sp.c_begin;
    row_base = (int64_t)n * p.T;
    seq_len = p.T;
    rec0 = sp.rec + ((int64_t)n * H + h) * (int64_t)sp.c_count * REC_BYTES;
    if (seg_g > 1) {
      // this segment's chunks, and where its state enters and leaves
      const int lo = seg * sp.seg_len, hi = lo + sp.seg_len < sp.c_count ? lo + sp.seg_len
                                                                          : sp.c_count;
      nc = hi > lo ? hi - lo : 0;
      c_first = lo;
      rec0 += (int64_t)lo * REC_BYTES;
      const int64_t seg_base =
          (((int64_t)n * seg_g + seg) * H + h) * (int64_t)DK * DV + half * 64;
      const int64_t next_base = seg_base + (int64_t)H * DK * DV;  // segment seg + 1
      if (sp.seg_pass == 1 && seg == 0) {   // segment 0 in full
        s_in = p.init_state;
        s_out = sp.seg_entry;
        out_base = next_base;
      } else if (sp.seg_pass == 1) {        // zero start (identity: below)
        s_in = nullptr;
        s_out = trans ? sp.seg_trans : sp.seg_s0;
        out_base = seg_base;
        emit = false;
      } else {                              // from its entry state, in full
        s_in = sp.seg_entry;
        in_base = seg_base;
        s_out = seg == seg_g - 1 ? p.final_state : nullptr;
      }
    }
  }
  // debug build: this chain's records and rows inside their buffers, else it
  // does nothing but report (every thread takes the same decision)
  bool dbg_bad = false;
  if (kda::kDebugChecks) {
    const int64_t first = nc > 0 ? (int64_t)(rec0 - sp.rec) / REC_BYTES : 0;
    dbg_bad = first < 0 || first + nc > sp.rec_items || row_base < 0 ||
              row_base + seq_len > sp.rows;
    if (dbg_bad) nc = 0;
  }

  uint64_t* bar_full = reinterpret_cast<uint64_t*>(smem + S_BAR);  // [2]
  uint64_t* bar_mma = bar_full + 2;
  uint64_t* bar_never = bar_full + 3;  // stall test only: nothing arrives on it
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + S_MISC);
  int* s_abort = reinterpret_cast<int*>(smem + S_MISC + 4);

  // record of chunk c and this half's V tile into stage c & 1 (V: one box of
  // 64 value channels x 64 rows from the input; rows past the sequence's end
  // are multiplied by zero columns of T Diag(beta))
  auto issue = [&](int c) {
    unsigned char* st = smem + (c & 1) * STAGE_BYTES;
    const unsigned char* src = rec0 + (int64_t)c * REC_BYTES;
    uint64_t* bar = bar_full + (c & 1);
    const int row = (int)(row_base + ((int64_t)c_first + c) * C);
    sm100::mbar_arrive_expect_tx(bar, ST_COPY + 512 + 8192);
    sm100::bulk_load(st + ST_KD, src + REC_KD, ST_COPY, bar);
    sm100::bulk_load(st + ST_GC, src + REC_GC, 512, bar);
    sm100::tma_load_3d(st + ST_V, &tm_v, bar, half * 64, h, row);
  };

  if (warp == 0) {
    sm100::tmem_alloc(s_tmem, S_TM_COLS);
    sm100::tmem_relinquish();
  }
  if (tid == 32) {
    sm100::mbar_init(bar_full, 1);
    sm100::mbar_init(bar_full + 1, 1);
    sm100::mbar_init(bar_mma, 1);
    sm100::mbar_init(bar_never, 1);
    sm100::fence_mbar_init();
    if (nc > 0) issue(0);
    if (nc > 1) issue(1);
  }
  if (tid == 0) *s_abort = 0;
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_q = 32u * (warp & 3);
  if (dbg_bad && tid == 0 && p.dev_status) atomicExch(p.dev_status, (int32_t)KDA_ERR_BOUNDS);

  // entry state into TMEM (lane = key channel); a transition run starts
  // from the identity's columns half * 64 ..
  if (warp < 4) {
    const int i = tid;
    for (int c = 0; c < 64; c += 16) {
      uint32_t r[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        r[e] = __float_as_uint(s_in && involved ? s_in[in_base + (int64_t)i * DV + c + e]
                               : (trans && i == half * 64 + c + e) ? 1.0f : 0.0f);
      sm100::tmem_st16(sm100::taddr(tmem, lane_q, TM_S + c), r);
    }
    sm100::tmem_wait_st();
  }

  uint32_t mma_phase = 0;
  bool mma_pending = false;
  bool u_open = false;           // thread 0: a U product not yet followed by a commit
  int issued = nc < 2 ? nc : 2;  // chunks whose record copy has been issued
  int landed = 0;                 // chunks whose record copy has been waited for
  // one thread waits for the products; the others meet it at the barrier
  auto wait_mma = [&]() {
    bool ok1 = true;
    if (tid == 0) {
      ok1 = sm100::mbar_wait(bar_mma, mma_phase & 1);
      if (!ok1) record_error(p, s_abort, KDA_ERR_TIMEOUT);
    }
    const bool ok = __syncthreads_and(ok1);
    if (ok) ++mma_phase;
    mma_pending = !ok;
    sm100::tc_fence_after();
  };
  auto sync_all = [&]() {
    sm100::tc_fence_before();
    __syncthreads();
    sm100::tc_fence_after();
  };
  // output rows of chunk c (warps 6-7: TMEM lanes 64..127 = rows 0..63)
  auto write_out = [&](int c) {
    const int r = tid - 192;
    const int64_t cs = ((int64_t)c_first + c) * C;
    const int L = (seq_len - cs) < C ? (int)(seq_len - cs) : C;
    float o[64];
#pragma unroll
    for (int c16 = 0; c16 < 64; c16 += 16) {
      float v[16];
      sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_P + 64 * (c & 1) + c16), v);
#pragma unroll
      for (int e = 0; e < 16; ++e) o[c16 + e] = v[e];
    }
    sm100::tmem_wait_ld();
    if (r < L) {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) +
                           ((row_base + cs + r) * H + h) * DV + half * 64;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const uint4 w = make_uint4(sm100::pack_bf16x2(o[8 * g], o[8 * g + 1]),
                                   sm100::pack_bf16x2(o[8 * g + 2], o[8 * g + 3]),
                                   sm100::pack_bf16x2(o[8 * g + 4], o[8 * g + 5]),
                                   sm100::pack_bf16x2(o[8 * g + 6], o[8 * g + 7]));
        *reinterpret_cast<uint4*>(dst + 8 * g) = w;
      }
    }
  };
  sync_all();
  SPLIT_MARK(16, mk);

  for (int c = 0; c < nc; ++c) {
    const int s = c & 1;
    const unsigned char* st = smem + s * STAGE_BYTES;
    const uint32_t tm_p = TM_P + 64 * s;
    const bool stall = (sp.stall_test & 2) && c == 0;
    if (!(stall ? sm100::mbar_wait(bar_never, 0, kStallTestNs)
                : sm100::mbar_wait(bar_full + s, (uint32_t)((c >> 1) & 1)))) {
      record_error(p, s_abort, KDA_ERR_TIMEOUT);
    } else {
      landed = c + 1;
      // U = [T Diag(beta); -] V of this half, while the CUDA cores copy S
      // (the P product's commit covers it); a transition run has U = 0
      if (tid == 0 && !trans) {
        const uint32_t idu = sm100::idesc_bf16(128, 64, 0, 1);
        const uint32_t s_t = sm100::smem_u32(st + ST_T);
        const uint32_t s_v = sm100::smem_u32(st + ST_V);
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
          sm100::mma_ss(tmem + TM_U, sm100::smem_desc(s_t + 256 * k, 128, 1024),
                        sm100::smem_desc_sw128(s_v + 2048 * k, 1024, 1024), idu, k > 0);
        u_open = true;
      }
    }
    SPLIT_MARK(17, mk);

    // (1) bf16 copy of S (B of the P product) and S <- gamma_C S ahead of the
    //     rank-64 update (all warps: lane = key channel, 32 columns each)
    {
      const int i = tid & 127, cb = (warp >> 2) * 32;
      const float gc = reinterpret_cast<const float*>(st + ST_GC)[i];
      float sv[32];
#pragma unroll
      for (int c16 = 0; c16 < 32; c16 += 16) {
        float v[16];
        sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_S + cb + c16), v);
#pragma unroll
        for (int e = 0; e < 16; ++e) sv[c16 + e] = v[e];
      }
      sm100::tmem_wait_ld();
#pragma unroll
      for (int jg = 0; jg < 4; ++jg)
        st8_bf16(smem + S_SB + mn_off(cb + 8 * jg, i, 1024), sv + 8 * jg);
#pragma unroll
      for (int c16 = 0; c16 < 32; c16 += 16) {
        uint32_t r[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(gc * sv[c16 + e]);
        sm100::tmem_st16(sm100::taddr(tmem, lane_q, TM_S + cb + c16), r);
      }
      sm100::tmem_wait_st();
    }
    sm100::fence_async_smem();
    sync_all();
    SPLIT_MARK(18, mk);
    // (checks right after a barrier: a flag raised after it needs a wait that
    // timed out, seconds after every thread has read it here)
    if (*s_abort) break;

    // (2) P = [W; Q gamma] S
    if (tid == 0) {
      const uint32_t idesc = sm100::idesc_bf16(128, 64, 1, 1);
      const uint32_t sa = sm100::smem_u32(st + ST_WQ);
      const uint32_t sb = sm100::smem_u32(smem + S_SB);
#pragma unroll
      for (int k = 0; k < DK / 16; ++k)
        sm100::mma_ss(tmem + tm_p, sm100::smem_desc(sa + k * 4096, 2048, 128),
                      sm100::smem_desc(sb + k * 2048, 1024, 128), idesc, k > 0);
      sm100::mma_commit(bar_mma);
      u_open = false;
    }
    mma_pending = true;
    // output rows of the previous chunk while the tensor cores work on P
    if (emit && warp >= 6 && c > 0) write_out(c - 1);
    wait_mma();
    SPLIT_MARK(19, mk);

    // (3) Delta = U - W S (warps 0, 1, 4, 5: lane = row, 32 columns each)
    if ((warp & 3) < 2) {
      const int r = (warp & 1) * 32 + lane, cb = (warp >> 2) * 32;
      float d[32];
#pragma unroll
      for (int c16 = 0; c16 < 32; c16 += 16) {
        float v[16], u[16];
        sm100::tmem_ld16(sm100::taddr(tmem, lane_q, tm_p + cb + c16), v);
        sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_U + cb + c16), u);
        sm100::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) d[c16 + e] = trans ? -v[e] : u[e] - v[e];
      }
#pragma unroll
      for (int g = 0; g < 4; ++g)
        st8_bf16(smem + S_DL + mn_off(cb + 8 * g, r, 1024), d + 8 * g);
    }
    sm100::fence_async_smem();
    sync_all();
    SPLIT_MARK(20, mk);
    if (*s_abort) break;

    // (4) S += (K dec)^T Delta;  O = Q gamma S + A_qk Delta (rows 64.. of P;
    //     the A operand [-; A_qk] starts 8 KiB before A_qk, inside K dec, and
    //     its unused product rows land on the consumed W S rows)
    if (tid == 0) {
      const uint32_t id = sm100::idesc_bf16(128, 64, 0, 1);
      const uint32_t s_kd = sm100::smem_u32(st + ST_KD);
      const uint32_t s_x = sm100::smem_u32(st + ST_AQ - 8192);
      const uint32_t s_dl = sm100::smem_u32(smem + S_DL);
#pragma unroll
      for (int k = 0; k < C / 16; ++k)
        sm100::mma_ss(tmem + TM_S, sm100::smem_desc(s_kd + 256 * k, 128, 1024),
                      sm100::smem_desc(s_dl + k * 2048, 1024, 128), id, 1);
#pragma unroll
      for (int k = 0; k < C / 16; ++k)
        sm100::mma_ss(tmem + tm_p, sm100::smem_desc(s_x + 256 * k, 128, 1024),
                      sm100::smem_desc(s_dl + k * 2048, 1024, 128), id, 1);
      sm100::mma_commit(bar_mma);
    }
    mma_pending = true;
    wait_mma();
    SPLIT_MARK(21, mk);
    if (*s_abort) break;
    // the stage has been read for the last time: the record two chunks ahead
    if (c + 2 < nc) {
      if (tid == 32) issue(c + 2);
      issued = c + 3;
    }

    // (5) state checkpoint (all warps: lane = key channel, the 32 columns
    //     this warp rescales next, so program order alone keeps the read
    //     ahead of the next chunk's rescaling)
    if (p.ckpt && emit) {
      const int64_t cs = ((int64_t)c_first + c) * C;
      const int L = (seq_len - cs) < C ? (int)(seq_len - cs) : C;
      const int64_t done = cs + L;
      if (L == C && done % p.ckpt_every == 0 && done / p.ckpt_every <= p.ckpt_max) {
        const int i = tid & 127, cb = (warp >> 2) * 32;
        float* dst = p.ckpt + ((((int64_t)n * H + h) * p.ckpt_max + done / p.ckpt_every - 1) *
                                   DK + i) * DV + half * 64 + cb;
#pragma unroll
        for (int c16 = 0; c16 < 32; c16 += 16) {
          float v[16];
          sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_S + cb + c16), v);
          sm100::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(dst + c16 + e) =
                make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
      }
    }
    SPLIT_MARK(22, mk);
  }

  if (*s_abort || dbg_bad) {
    // bounded waits for copies and products still in flight (a U product
    // that no commit follows gets one first)
    if (tid == 0 && u_open) {
      sm100::mma_commit(bar_mma);
      mma_pending = true;
    }
    if (mma_pending) sm100::mbar_wait(bar_mma, mma_phase & 1, 200000000ull);
    for (int k = landed; k < issued; ++k)
      sm100::mbar_wait(bar_full + (k & 1), (uint32_t)((k >> 1) & 1), 200000000ull);
  } else {
    if (emit && nc > 0 && warp >= 6) write_out(nc - 1);
    if (s_out && involved && warp < 4) {
      const int i = tid;
      float* dst = s_out + out_base + (int64_t)i * DV;
      for (int c16 = 0; c16 < 64; c16 += 16) {
        float v[16];
        sm100::tmem_ld16(sm100::taddr(tmem, lane_q, TM_S + c16), v);
        sm100::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(dst + c16 + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
    }
  }
  sm100::tc_fence_before();
  __syncthreads();
  if (warp == 0) sm100::tmem_dealloc(tmem, S_TM_COLS);
}

// Entry states of the segments of a dense batch, in order: entry[s + 1] =
// trans[s] entry[s] + s0[s] for s = 1 .. G - 2 (entry[1] is segment 0's
// final state), the state update of a span being affine in the state that
// enters it.  fp32 on the CUDA cores; grid (H, N, DV / 32), 256 threads:
// thread = (key row i, 16 of the block's 32 value columns).
constexpr int SEG_SC = 32, SEG_LDP = DK + 1;
static_assert(DK == DV, "a transition is stored in a state's layout");
constexpr int SEG_SMEM = (int)sizeof(float) * (DK * SEG_LDP + DK * SEG_SC);
__global__ void __launch_bounds__(256)
    kda_split_seg_entries_kernel(const float* trans, const float* s0, float* entry, int N,
                                 int H, int G) {
  extern __shared__ float sm_f[];
  float* sP = sm_f;                 // [DK][SEG_LDP]
  float* sS = sP + DK * SEG_LDP;    // [DK][SEG_SC]
  const int h = blockIdx.x, n = blockIdx.y, c0 = blockIdx.z * SEG_SC;
  const int tid = threadIdx.x, i = tid & (DK - 1), cg = (tid >> 7) * 16;
  auto at = [&](int sg) { return (((int64_t)n * G + sg) * H + h) * (int64_t)DK * DV; };
  for (int e = tid; e < DK * SEG_SC; e += 256)
    sS[e] = entry[at(1) + (int64_t)(e / SEG_SC) * DV + c0 + e % SEG_SC];
  for (int sg = 1; sg + 1 < G; ++sg) {
    const float* P = trans + at(sg);  // [DK][DK] (DK == DV)
    __syncthreads();
    for (int e = tid; e < DK * DK; e += 256) sP[(e / DK) * SEG_LDP + e % DK] = P[e];
    __syncthreads();
    float acc[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] = s0[at(sg) + (int64_t)i * DV + c0 + cg + c];
    for (int k = 0; k < DK; ++k) {
      const float pv = sP[i * SEG_LDP + k];
#pragma unroll
      for (int c = 0; c < 16; ++c) acc[c] = fmaf(pv, sS[k * SEG_SC + cg + c], acc[c]);
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      sS[i * SEG_SC + cg + c] = acc[c];
      entry[at(sg + 1) + (int64_t)i * DV + c0 + cg + c] = acc[c];
    }
  }
}

// ===========================================================================
// packed batches: the chunk columns of the sequences
// ===========================================================================
// The order in which the state CTAs take the sequences: longest first.  A
// sequence's chain is the longest single piece of work of the state pass,
// and the CTAs start in grid order, so a long sequence placed last would run
// on alone at the end.  order[rank] = n with rank = the number of sequences
// with more chunks, or as many and a lower index (a permutation, also for
// the all-zero offsets of a malformed batch); beyond kOrderMax sequences
// the count of comparisons is not worth it and the order is the identity.
constexpr int kOrderMax = 8192;
__global__ void __launch_bounds__(256)
    kda_split_order_kernel(const int* off, int N, int* order) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  if (N > kOrderMax) {
    order[n] = n;
    return;
  }
  const int c = off[n + 1] - off[n];
  int rank = 0;
  for (int m = 0; m < N; ++m) {
    const int cm = off[m + 1] - off[m];
    rank += (cm > c || (cm == c && m < n)) ? 1 : 0;
  }
  order[rank] = n;
}

// One CTA: off[n] = chunks of the sequences before n (an exclusive scan of
// ceil(len / 64)), off[N] = their total.  Malformed offsets (cu[0] != 0,
// cu[N] != T, a decreasing pair) are reported through the status word and
// leave every sequence without chunks.
__global__ void __launch_bounds__(1024)
    kda_split_offsets_kernel(const int32_t* cu, int N, int T, int* off, int32_t* dev_status) {
  __shared__ int s_bad, s_carry, s_warp[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_bad = (cu[0] != 0 || cu[N] != T) ? 1 : 0;
    s_carry = 0;
  }
  __syncthreads();
  for (int base = 0; base < N; base += 1024) {
    const int n = base + tid;
    int cnt = 0;
    if (n < N) {
      const int len = cu[n + 1] - cu[n];
      if (len < 0) s_bad = 1;  // (every writer stores the same value)
      else cnt = (len + C - 1) / C;
    }
    int x = cnt;  // inclusive scan: within the warp, then over the warps
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int wv = s_warp[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wv, d);
        if (lane >= d) wv += y;
      }
      s_warp[lane] = wv;
    }
    __syncthreads();
    if (n < N) off[n] = s_carry + (warp ? s_warp[warp - 1] : 0) + x - cnt;
    __syncthreads();
    if (tid == 0) s_carry += s_warp[31];
    __syncthreads();
  }
  if (s_bad) {
    for (int n = tid; n <= N; n += 1024) off[n] = 0;
    if (tid == 0 && dev_status) atomicExch(dev_status, (int32_t)KDA_ERR_BAD_SEQLENS);
  } else if (tid == 0) {
    off[N] = s_carry;
  }
}

// tab[g] for every chunk column g < g_max: {first token row, n | rows << 24}
// of the chunk there ({0, 0} past the last one); n by bisection over off
__global__ void kda_split_table_kernel(const int32_t* cu, const int* off, int N, int g_max,
                                       int2* tab) {
  const int total = off[N];
  for (int g = blockIdx.x * blockDim.x + threadIdx.x; g < g_max; g += gridDim.x * blockDim.x) {
    int2 e = make_int2(0, 0);
    if (g < total) {
      int lo = 0, hi = N - 1;  // the last n with off[n] <= g
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= g) lo = mid;
        else hi = mid - 1;
      }
      const int cl = g - off[lo];
      const int len = cu[lo + 1] - cu[lo];
      const int L = len - cl * C < C ? len - cl * C : C;
      e = make_int2(cu[lo] + cl * C, lo | (L << 24));
    }
    tab[g] = e;
  }
}

// the stall test's flags for the next calls (test hook, see SplitParams)
std::atomic<int> g_stall_test{0};
// debug builds: records the kernels are told the workspace holds (0: real)
std::atomic<long long> g_record_capacity{0};
int64_t told_capacity(int64_t real) {
  const long long o = g_record_capacity.load();
  return o > 0 && o < real ? o : real;
}

// default bytes of records held at once (the slice length follows from it):
// a dense batch's slices, and a packed batch's (whose sequences end at
// different chunk columns, so each slice waits for its longest chain: one
// slice is best, 12.1 against 13.4 ms for a 1M-token batch of 28 sequences
// in five)
constexpr size_t kRecordBudget = (size_t)4 << 30;
constexpr size_t kPackedRecordBudget = (size_t)32 << 30;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
size_t carry_bytes(int N, int H) { return align256((size_t)N * H * DK * DV * sizeof(float)); }

// packed batches: [carry][chunk_off: N + 1 ints][seq_order: N ints]
// [chunk_tab: g_max entries][records: H x the chunk columns of one slice]
int packed_g_max(int N, int T) { return (int)(((int64_t)T + C - 1) / C + N); }
struct PackedLayout {
  size_t off_at, ord_at, tab_at, rec_at, total;
};
PackedLayout packed_layout(int N, int T, int H, int64_t cols) {
  PackedLayout L;
  const size_t g = (size_t)packed_g_max(N, T);
  L.off_at = carry_bytes(N, H);
  L.ord_at = L.off_at + align256((size_t)(N + 1) * sizeof(int));
  L.tab_at = L.ord_at + align256((size_t)N * sizeof(int));
  L.rec_at = L.tab_at + align256(g * sizeof(int2));
  L.total = L.rec_at + (size_t)cols * H * REC_BYTES;
  return L;
}
// Segments of a dense batch on the two-kernel path.  When its state chains
// (2 N H CTAs) leave most SMs idle and its sequences are long, each sequence
// is cut into G segments: pass 1 runs segment 0 in full and, beside it,
// summarises segments 1 .. G - 2 (zero-start final state and cumulative
// transition: four state CTAs each); the entry states follow by the
// composition rule; pass 2 reruns segments 1 .. G - 1 from them.  The
// chain a pass runs is one segment long, so the time goes from about T to
// 2 T / G chunk steps.  G is the most that keeps pass 1 in one wave of state
// CTAs (one per SM), with at least 128 chunks per segment, and the records
// of every chunk (read by both passes) within a budget.
constexpr size_t kSegRecordBudget = (size_t)32 << 30;
constexpr int kSegMinChunks = 128;
// test hook: > 0 forces that many segments where the sizes allow, < 0
// turns segments off, 0 chooses by the rule above
std::atomic<int> g_force_segments{0};
int split_segments(int N, int T, int H, int sms) {
  const int64_t nchunks = ((int64_t)T + C - 1) / C;
  const int64_t nh = (int64_t)N * H;
  const int forced = g_force_segments.load();
  int64_t G;
  if (forced < 0) return 1;
  if (forced > 0) {
    G = forced;
  } else {
    if (6 * nh > sms) return 1;
    G = 2 + (sms - 2 * nh) / (4 * nh);
    if (G > nchunks / kSegMinChunks) G = nchunks / kSegMinChunks;
    if (G < 3 || nh * nchunks * (int64_t)REC_BYTES > (int64_t)kSegRecordBudget) return 1;
  }
  // every segment holds at least one chunk: (G - 1) ceil(nchunks / G) < nchunks
  while (G > 2 && (G - 1) * ((nchunks + G - 1) / G) >= nchunks) --G;
  if (G < 3 || (int64_t)N * G > 65535 || 2 + 4 * (G - 2) > 65535) return 1;
  return (int)G;
}
int seg_chunks(int T, int G) {
  const int64_t nchunks = ((int64_t)T + C - 1) / C;
  return (int)((nchunks + G - 1) / G);
}
// [carry][records of every chunk][entry states][zero-start states][transitions]
size_t seg_state_bytes(int N, int H, int G) {
  return align256((size_t)N * G * H * DK * DV * sizeof(float));
}
size_t split_seg_workspace_bytes(int N, int T, int H, int G) {
  const int64_t nchunks = ((int64_t)T + C - 1) / C;
  return carry_bytes(N, H) + (size_t)N * H * REC_BYTES * (size_t)nchunks +
         3 * seg_state_bytes(N, H, G);
}

// chunk columns per slice of the default workspace: all of them while their
// records fit in the record budget
int64_t packed_default_cols(int N, int T, int H) {
  const int64_t g = packed_g_max(N, T);
  int64_t fit = (int64_t)(kPackedRecordBudget / ((size_t)H * REC_BYTES));
  if (fit < 1) fit = 1;
  return g < fit ? g : fit;
}

}  // namespace

// Device bytes of the two-kernel path for a packed batch of T tokens in N
// sequences: by default the chunk records of every column while they fit in
// the record budget (else slices of columns); at least one column's records.
size_t kda_split_packed_workspace_bytes(int N, int T, int H) {
  if (N < 1 || H < 1 || T < 1) return 0;
  return packed_layout(N, T, H, packed_default_cols(N, T, H)).total;
}
size_t kda_split_packed_min_workspace_bytes(int N, int T, int H) {
  if (N < 1 || H < 1 || T < 1) return 0;
  return packed_layout(N, T, H, 1).total;
}

#ifdef KDA_PHASE_TIMING
extern "C" int kda_split_timing_read(unsigned long long* out32, int reset) {
  if (cudaMemcpyFromSymbol(out32, kda_split_cycles, sizeof(unsigned long long) * 32) !=
      cudaSuccess)
    return -1;
  if (reset) {
    unsigned long long z[32] = {0};
    cudaMemcpyToSymbol(kda_split_cycles, z, sizeof(z));
  }
  return 0;
}
#endif

// Device bytes of the two-kernel path: the state carried between slices,
// then the records of one slice.  The default holds up to 4 GiB of records;
// the minimum holds one chunk's records per (sequence, head).
size_t kda_split_workspace_bytes(int N, int T, int H) {
  if (N < 1 || H < 1 || T < 1) return 0;
  const int G = split_segments(N, T, H, kda_device_sms());
  if (G > 1) return split_seg_workspace_bytes(N, T, H, G);
  const int64_t nchunks = ((int64_t)T + C - 1) / C;
  const size_t per = (size_t)N * H * REC_BYTES;
  int64_t slice = (int64_t)(kRecordBudget / per);
  if (slice < 1) slice = 1;
  if (slice > nchunks) slice = nchunks;
  return carry_bytes(N, H) + per * (size_t)slice;
}
size_t kda_split_min_workspace_bytes(int N, int H) {
  if (N < 1 || H < 1) return 0;
  return carry_bytes(N, H) + (size_t)N * H * REC_BYTES;
}

namespace {

// What every slice launch of one call shares: the tensor maps over the
// inputs, the SM count, and where the records and the carried state live.
struct SplitPlan {
  CUtensorMap mq, mk, mg, mv;  // mv: V, 128-byte swizzled (state kernel)
  int sms = 0;
  int nchunks = 0;
  size_t carry = 0, per = 0;   // bytes: carried state; records of one chunk column
  size_t fit = 0;              // chunk columns the workspace holds
  float* through = nullptr;    // state between slices
  unsigned char* rec = nullptr;
  // packed batches
  bool packed = false;
  int g_max = 0;
  int* chunk_off = nullptr;
  int* seq_order = nullptr;
  int2* chunk_tab = nullptr;
};

kda_status plan_split(const kda::FwdParams& p, void* workspace, size_t workspace_bytes,
                      SplitPlan& pl) {
  pl.packed = p.cu_seqlens != nullptr;
  if (p.dk != DK || p.dv != DV || p.T < 1) return KDA_ERR_UNSUPPORTED;
  if (p.N > 65535 || p.H > 65535) return KDA_ERR_UNSUPPORTED;
  const int64_t rows = pl.packed ? (int64_t)p.T : (int64_t)p.N * p.T;
  if (rows >= (int64_t)1 << 31) return KDA_ERR_UNSUPPORTED;
  if (((uintptr_t)workspace & 255) != 0) return KDA_ERR_MISALIGNED;
  pl.carry = carry_bytes(p.N, p.H);
  if (pl.packed) {
    const PackedLayout L = packed_layout(p.N, p.T, p.H, 1);
    if (workspace_bytes < L.total) return KDA_ERR_WORKSPACE;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    pl.g_max = packed_g_max(p.N, p.T);
    pl.chunk_off = reinterpret_cast<int*>(ws + L.off_at);
    pl.seq_order = reinterpret_cast<int*>(ws + L.ord_at);
    pl.chunk_tab = reinterpret_cast<int2*>(ws + L.tab_at);
    pl.per = (size_t)p.H * REC_BYTES;  // records of one chunk column
    pl.fit = (workspace_bytes - L.rec_at) / pl.per;
  } else {
    pl.per = (size_t)p.N * p.H * REC_BYTES;
    if (workspace_bytes < pl.carry + pl.per) return KDA_ERR_WORKSPACE;
    pl.nchunks = (int)(((int64_t)p.T + C - 1) / C);
    pl.fit = (workspace_bytes - pl.carry) / pl.per;
  }
  pl.sms = kda_device_sms();
  if (pl.sms < 1) return KDA_ERR_CUDA;
  // unswizzled tiles: every read of them goes along one row
  if (!make_map(&pl.mq, p.q, rows, p.H, DK, false) || !make_map(&pl.mk, p.k, rows, p.H, DK, false) ||
      !make_map(&pl.mg, p.g, rows, p.H, DK, false) ||
      !make_map(&pl.mv, p.v, rows, p.H, DV, true))
    return KDA_ERR_CUDA;
  if (kda_smem_attr((const void*)kda_tc_intra_kernel, I_SMEM) != KDA_OK ||
      kda_smem_attr((const void*)kda_tc_state_kernel, S_SMEM) != KDA_OK)
    return KDA_ERR_CUDA;
  // the state crosses slices in final_state when there is one (each CTA
  // reads its part before it writes it), else in the workspace
  pl.through = p.final_state ? p.final_state : static_cast<float*>(workspace);
  if (pl.packed) {
    pl.rec = static_cast<unsigned char*>(workspace) + packed_layout(p.N, p.T, p.H, 1).rec_at;
    return KDA_OK;
  }
  pl.rec = static_cast<unsigned char*>(workspace) + pl.carry;
  return KDA_OK;
}

// One slice, chunks [c0, c0 + cnt) of every sequence: the intra kernel over
// it (on `s_intra`, at most `grid_cap` CTAs), then the state kernel (on
// `s_state`), the records at `rec`.  `stages` selects the kernels (bit 0
// intra, bit 1 state).
kda_status launch_slice(const kda::FwdParams& p, const SplitPlan& pl, int c0, int cnt,
                        cudaStream_t s_intra, cudaStream_t s_state, int stages,
                        unsigned char* rec, int grid_cap, int rec_stride = 0) {
  SplitParams sp{};
  sp.p = p;
  sp.rec = rec;
  sp.c_begin = c0;
  sp.c_count = cnt;
  sp.chunk_tab = nullptr;
  sp.chunk_off = nullptr;
  sp.g_max = 0;
  sp.g_begin = 0;
  sp.g_count = 0;
  sp.s_in = c0 == 0 ? p.init_state : pl.through;
  sp.s_out = c0 + cnt == pl.nchunks ? p.final_state : pl.through;
  sp.stall_test = g_stall_test.load();
  sp.rec_items = told_capacity((int64_t)p.N * p.H * (rec_stride > 0 ? rec_stride : cnt));
  sp.rows = (int64_t)p.N * p.T;
  sp.rec_stride = rec_stride;
  if (stages & 1) {
    // persistent: two CTAs per SM walk the slice's (sequence, head, chunk) items
    const int64_t items = (int64_t)p.N * p.H * cnt;
    const int grid = items < (int64_t)grid_cap ? (int)items : grid_cap;
    kda_tc_intra_kernel<<<grid, kThreads, I_SMEM, s_intra>>>(pl.mq, pl.mk, pl.mg, sp);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
  }
  if (stages & 2) {
    kda_tc_state_kernel<<<dim3(2, p.H, p.N), kThreads, S_SMEM, s_state>>>(pl.mv, sp);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

// Streams and events of the overlapped slice schedule, created once per
// device (the state stream at the highest priority, so that its CTAs are
// placed first) and used under one lock for a call's whole enqueue sequence.
struct OverlapRes {
  cudaStream_t s_intra = nullptr, s_state = nullptr;
  cudaEvent_t ev_start = nullptr, ev_intra[2] = {}, ev_state[2] = {};
};
std::mutex g_ov_mu;
std::map<int, OverlapRes> g_ov;

// (called with g_ov_mu held)
kda_status overlap_res(OverlapRes** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  auto it = g_ov.find(dev);
  if (it != g_ov.end()) {
    *out = &it->second;
    return KDA_OK;
  }
  OverlapRes r;
  int least = 0, greatest = 0;
  bool ok = cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess &&
            cudaStreamCreateWithPriority(&r.s_intra, cudaStreamNonBlocking, least) ==
                cudaSuccess &&
            cudaStreamCreateWithPriority(&r.s_state, cudaStreamNonBlocking, greatest) ==
                cudaSuccess &&
            cudaEventCreateWithFlags(&r.ev_start, cudaEventDisableTiming) == cudaSuccess;
  for (int b = 0; b < 2 && ok; ++b)
    ok = cudaEventCreateWithFlags(&r.ev_intra[b], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&r.ev_state[b], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) return KDA_ERR_CUDA;
  *out = &(g_ov[dev] = r);
  return KDA_OK;
}

// Slices of a dense batch whose state chains leave most SMs idle (few
// sequence x head pairs, long sequences): slice i + 1's intra kernel runs on
// the SMs the state CTAs leave free while slice i's state pass runs, the
// records alternating between the two halves of the record buffer.  The
// kernels never wait on one another: the library's two streams order them
// by events (slice i's state after its intra kernel; slice i + 2's intra
// kernel after slice i's state pass has read that half).  The result is the
// same as one slice after another.
kda_status run_overlapped(const kda::FwdParams& p, const SplitPlan& pl, int slice,
                          cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_ov_mu);
  OverlapRes* r = nullptr;
  kda_status st = overlap_res(&r);
  if (st != KDA_OK) return st;
  const int state_ctas = 2 * p.N * p.H;
  const int cap_alone = 2 * pl.sms, cap_beside = 2 * (pl.sms - state_ctas);
  unsigned char* half[2] = {pl.rec, pl.rec + pl.per * (size_t)slice};
  auto cu = [&](cudaError_t e) {
    if (e != cudaSuccess && st == KDA_OK) st = KDA_ERR_CUDA;
  };
  cu(cudaEventRecord(r->ev_start, stream));
  cu(cudaStreamWaitEvent(r->s_intra, r->ev_start, 0));
  cu(cudaStreamWaitEvent(r->s_state, r->ev_start, 0));
  int last = 0;
  for (int i = 0, c0 = 0; c0 < pl.nchunks && st == KDA_OK; ++i, c0 += slice) {
    const int b = i & 1, cnt = pl.nchunks - c0 < slice ? pl.nchunks - c0 : slice;
    if (i >= 2) cu(cudaStreamWaitEvent(r->s_intra, r->ev_state[b], 0));
    if (st == KDA_OK)
      st = launch_slice(p, pl, c0, cnt, r->s_intra, r->s_state, 1, half[b],
                        i == 0 ? cap_alone : cap_beside);
    cu(cudaEventRecord(r->ev_intra[b], r->s_intra));
    cu(cudaStreamWaitEvent(r->s_state, r->ev_intra[b], 0));
    if (st == KDA_OK)
      st = launch_slice(p, pl, c0, cnt, r->s_intra, r->s_state, 2, half[b], cap_alone);
    cu(cudaEventRecord(r->ev_state[b], r->s_state));
    last = b;
  }
  // the caller's stream continues once the last state pass is done (which
  // follows every intra kernel)
  cu(cudaStreamWaitEvent(stream, r->ev_state[last], 0));
  return st;
}

// A packed batch's chunk table: the sequences' chunk offsets, then the first
// row and row count of every column.
kda_status packed_prepare(const kda::FwdParams& p, const SplitPlan& pl, cudaStream_t stream) {
  kda_split_offsets_kernel<<<1, 1024, 0, stream>>>(p.cu_seqlens, p.N, p.T, pl.chunk_off,
                                                   p.dev_status);
  kda_split_order_kernel<<<(p.N + 255) / 256, 256, 0, stream>>>(pl.chunk_off, p.N,
                                                                pl.seq_order);
  const int tb_need = (pl.g_max + 255) / 256;
  const int tb = tb_need < 8 * pl.sms ? tb_need : 8 * pl.sms;
  kda_split_table_kernel<<<tb, 256, 0, stream>>>(p.cu_seqlens, pl.chunk_off, p.N, pl.g_max,
                                                 pl.chunk_tab);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// Both kernels over chunk columns [g0, g0 + cnt) of a packed batch (after
// packed_prepare), the records at the start of the workspace's record area.
kda_status packed_slice(const kda::FwdParams& p, const SplitPlan& pl, int g0, int cnt,
                      cudaStream_t stream) {
  SplitParams sp{};
  sp.p = p;
  sp.rec = pl.rec;
  sp.c_begin = 0;
  sp.c_count = 0;
  // sequences start from init_state and end in final_state; one that
  // spans slices carries its state through final_state or the workspace
  sp.s_in = pl.through;
  sp.s_out = pl.through;
  sp.chunk_tab = pl.chunk_tab;
  sp.chunk_off = pl.chunk_off;
  sp.seq_order = pl.seq_order;
  sp.g_max = pl.g_max;
  sp.g_begin = g0;
  sp.g_count = cnt;
  sp.stall_test = g_stall_test.load();
  sp.rec_items = told_capacity((int64_t)cnt * p.H);
  sp.rows = p.T;
  const int64_t items = (int64_t)cnt * p.H;
  const int grid = items < 2 * (int64_t)pl.sms ? (int)items : 2 * pl.sms;
  kda_tc_intra_kernel<<<grid, kThreads, I_SMEM, stream>>>(pl.mq, pl.mk, pl.mg, sp);
  if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
  kda_tc_state_kernel<<<dim3(2, p.H, p.N), kThreads, S_SMEM, stream>>>(pl.mv, sp);
  if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
  return KDA_OK;
}

// The slices run back to back on `stream`.
// A packed batch: its chunk table, then both kernels over each slice of
// chunk columns in turn (one slice when the workspace holds every column).
kda_status launch_packed(const kda::FwdParams& p, const SplitPlan& pl, cudaStream_t stream) {
  kda_status st = packed_prepare(p, pl, stream);
  const int fit = pl.fit < (size_t)pl.g_max ? (int)pl.fit : pl.g_max;
  for (int g0 = 0; g0 < pl.g_max && st == KDA_OK; g0 += fit)
    st = packed_slice(p, pl, g0, pl.g_max - g0 < fit ? pl.g_max - g0 : fit, stream);
  return st;
}

// A dense batch in G segments (see split_segments): the records of segments
// 0 .. G - 2, then pass 1 (segment 0 in full, the summaries of segments
// 1 .. G - 2) and the entry states, while the last segment's records are
// made on the SMs pass 1 leaves free; then pass 2 (segments 1 .. G - 1 in
// full).  The kernels never wait on one another: the library's two streams
// order them by events (as in the overlapped slice schedule; one stream
// while the caller's stream is being captured).  The workspace holds
// split_seg_workspace_bytes(N, T, H, G).
kda_status run_split_segmented(const kda::FwdParams& p, const SplitPlan& pl, void* workspace,
                               int G, cudaStream_t stream) {
  const int L = seg_chunks(p.T, G), head = (G - 1) * L;  // chunks pass 1 reads
  if (kda_smem_attr((const void*)kda_split_seg_entries_kernel, SEG_SMEM) != KDA_OK)
    return KDA_ERR_CUDA;
  float* seg = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) +
                                        carry_bytes(p.N, p.H) +
                                        (size_t)p.N * p.H * REC_BYTES * (size_t)pl.nchunks);
  const size_t per = seg_state_bytes(p.N, p.H, G) / sizeof(float);
  SplitParams sp{};
  sp.p = p;
  sp.rec = pl.rec;
  sp.c_begin = 0;
  sp.c_count = pl.nchunks;
  sp.stall_test = g_stall_test.load();
  sp.rec_items = told_capacity((int64_t)p.N * p.H * pl.nchunks);
  sp.rows = (int64_t)p.N * p.T;
  sp.seg_g = G;
  sp.seg_len = L;
  sp.seg_entry = seg;
  sp.seg_s0 = seg + per;
  sp.seg_trans = seg + 2 * per;
  const int pass1 = (2 + 4 * (G - 2)) * p.H * p.N;  // state CTAs of pass 1
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  const bool side = cudaStreamIsCapturing(stream, &cap) == cudaSuccess &&
                    cap == cudaStreamCaptureStatusNone && pass1 < pl.sms;
  std::unique_lock<std::mutex> lock(g_ov_mu, std::defer_lock);
  OverlapRes* r = nullptr;
  if (side) {
    lock.lock();
    if (overlap_res(&r) != KDA_OK) return KDA_ERR_CUDA;
  }
  kda_status st = KDA_OK;
  auto cu = [&](cudaError_t e) {
    if (e != cudaSuccess && st == KDA_OK) st = KDA_ERR_CUDA;
  };
  // records of segments 0 .. G - 2 on the caller's stream
  st = launch_slice(p, pl, 0, head, stream, stream, 1, pl.rec, 2 * pl.sms, pl.nchunks);
  cudaStream_t s_state = stream, s_intra = stream;
  if (side && st == KDA_OK) {
    s_state = r->s_state;
    s_intra = r->s_intra;
    cu(cudaEventRecord(r->ev_start, stream));
    cu(cudaStreamWaitEvent(s_state, r->ev_start, 0));
    cu(cudaStreamWaitEvent(s_intra, r->ev_start, 0));
  }
  if (st == KDA_OK) {
    sp.seg_pass = 1;
    kda_tc_state_kernel<<<dim3(2 + 4 * (G - 2), p.H, p.N), kThreads, S_SMEM, s_state>>>(pl.mv,
                                                                                       sp);
    cu(cudaGetLastError());
  }
  if (st == KDA_OK) {
    kda_split_seg_entries_kernel<<<dim3(p.H, p.N, DV / SEG_SC), 256, SEG_SMEM, s_state>>>(
        sp.seg_trans, sp.seg_s0, sp.seg_entry, p.N, p.H, G);
    cu(cudaGetLastError());
  }
  // the last segment's records beside pass 1 (its CTAs take whole SMs)
  if (st == KDA_OK) {
    const int cap_beside = side ? 2 * (pl.sms - pass1) : 2 * pl.sms;
    st = launch_slice(p, pl, head, pl.nchunks - head, s_intra, s_intra, 1, pl.rec, cap_beside,
                      pl.nchunks);
  }
  if (side) {
    cu(cudaEventRecord(r->ev_intra[0], s_intra));
    cu(cudaStreamWaitEvent(s_state, r->ev_intra[0], 0));
  }
  if (st == KDA_OK) {
    sp.seg_pass = 2;
    kda_tc_state_kernel<<<dim3(2 * (G - 1), p.H, p.N), kThreads, S_SMEM, s_state>>>(pl.mv, sp);
    cu(cudaGetLastError());
  }
  if (side) {
    // the caller's stream continues once pass 2 is done (which follows
    // every other launch of the call)
    cu(cudaEventRecord(r->ev_state[0], s_state));
    cu(cudaStreamWaitEvent(stream, r->ev_state[0], 0));
  }
  return st;
}

kda_status run_split(const kda::FwdParams& p, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream, int stages, bool one_slice) {
  SplitPlan pl;
  kda_status st = plan_split(p, workspace, workspace_bytes, pl);
  if (st != KDA_OK) return st;
  if (pl.packed) return stages == 3 ? launch_packed(p, pl, stream) : KDA_ERR_UNSUPPORTED;
  const int slice = pl.fit < (size_t)pl.nchunks ? (int)pl.fit : pl.nchunks;
  if (one_slice && slice < pl.nchunks) return KDA_ERR_WORKSPACE;
  // few long chains and room for every record: segments
  if (stages == 3 && !one_slice && !p.ckpt) {
    const int G = split_segments(p.N, p.T, p.H, pl.sms);
    if (G > 1 && workspace_bytes >= split_seg_workspace_bytes(p.N, p.T, p.H, G))
      return run_split_segmented(p, pl, workspace, G, stream);
  }
  // more than one slice and state chains on at most half of the SMs: the
  // overlapped schedule (not while the caller's stream is being captured)
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (stages == 3 && !one_slice && slice < pl.nchunks && pl.fit >= 2 &&
      4 * (int64_t)p.N * p.H <= pl.sms &&
      cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusNone)
    return run_overlapped(p, pl, (int)(pl.fit / 2), stream);
  for (int c0 = 0; c0 < pl.nchunks && st == KDA_OK; c0 += slice)
    st = launch_slice(p, pl, c0, pl.nchunks - c0 < slice ? pl.nchunks - c0 : slice, stream,
                      stream, stages, pl.rec, 2 * pl.sms);
  return st;
}

}  // namespace

kda_status kda_run_split(const kda::FwdParams& p, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
  return run_split(p, workspace, workspace_bytes, stream, 3, false);
}

// Chunks [c0, c0 + cnt) alone (both kernels); the state enters from
// init_state (c0 = 0) or from where the previous range left it, and leaves
// into final_state (last range) or that carry.  The workspace must hold cnt
// chunk columns of records.
kda_status kda_run_split_range(const kda::FwdParams& p, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream, int c0, int cnt) {
  if (p.cu_seqlens) return KDA_ERR_UNSUPPORTED;
  SplitPlan pl;
  kda_status st = plan_split(p, workspace, workspace_bytes, pl);
  if (st != KDA_OK) return st;
  if (c0 < 0 || cnt < 1 || c0 + cnt > pl.nchunks || (size_t)cnt > pl.fit) return KDA_ERR_INVALID_ARG;
  return launch_slice(p, pl, c0, cnt, stream, stream, 3, pl.rec, 2 * pl.sms);
}

// Chunk columns [g0, g0 + cnt) of a packed batch alone (both kernels), the
// chunk table built first when `prepare` is set (the first range of a call).
// Sequences enter from init_state where they start, else from the state the
// previous range left in final_state or the workspace; the workspace must
// hold cnt columns of records.
kda_status kda_run_split_packed_range(const kda::FwdParams& p, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream, int g0,
                                      int cnt, bool prepare) {
  if (!p.cu_seqlens) return KDA_ERR_UNSUPPORTED;
  SplitPlan pl;
  kda_status st = plan_split(p, workspace, workspace_bytes, pl);
  if (st != KDA_OK) return st;
  if (g0 < 0 || cnt < 1 || g0 + cnt > pl.g_max || (size_t)cnt > pl.fit)
    return KDA_ERR_INVALID_ARG;
  if (prepare && (st = packed_prepare(p, pl, stream)) != KDA_OK) return st;
  return packed_slice(p, pl, g0, cnt, stream);
}

// Chunk columns of a packed batch: an upper bound, ceil(T / 64) + N.
int kda_split_packed_g_max(int N, int T) { return packed_g_max(N, T); }

// Device bytes of the two-kernel path for a packed batch run `cols` chunk
// columns at a time.
size_t kda_split_packed_slice_workspace_bytes(int N, int T, int H, int cols) {
  if (N < 1 || H < 1 || T < 1 || cols < 1) return 0;
  return packed_layout(N, T, H, cols).total;
}

// Device bytes of the two-kernel path for slices of `chunks` chunks.
size_t kda_split_slice_workspace_bytes(int N, int H, int chunks) {
  if (N < 1 || H < 1 || chunks < 1) return 0;
  return carry_bytes(N, H) + (size_t)N * H * REC_BYTES * (size_t)chunks;
}

extern "C" kda_status kda_split_stage(int stage, const uint16_t* q, const uint16_t* k,
                                      const uint16_t* v, const uint16_t* g_logit,
                                      const uint16_t* beta, const float* init_state,
                                      uint16_t* out, float* final_state, int B, int T, int H,
                                      float scale, void* workspace, size_t workspace_bytes,
                                      int32_t* dev_status, kda_stream_t stream) {
  if (stage != 1 && stage != 2) return KDA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || T < 1 || !q || !k || !v || !g_logit || !beta || !out || !workspace)
    return KDA_ERR_INVALID_ARG;
  const uintptr_t pa = (uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)g_logit |
                       (uintptr_t)out | (uintptr_t)init_state | (uintptr_t)final_state;
  if ((pa & 15) != 0 || ((uintptr_t)beta & 1) != 0) return KDA_ERR_MISALIGNED;
  kda::FwdParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g_logit; p.beta = beta;
  p.init_state = init_state; p.out = out; p.final_state = final_state;
  p.dev_status = dev_status;
  p.N = B; p.T = T; p.H = H; p.dk = DK; p.dv = DV; p.scale = scale;
  return run_split(p, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), stage,
                   true);
}

// Test hook: the next calls of the two-kernel path make their first wait in
// the intra kernel (flags bit 0) and / or the state kernel (bit 1) run out
// (see SplitParams::stall_test); 0 restores normal calls.
// Segments per sequence a dense bf16 call at dk = dv = 128 on the
// two-kernel path takes with this workspace (1: the plain form).
extern "C" int kda_split_segment_count(int N, int T, int H, size_t workspace_bytes) {
  if (N < 1 || H < 1 || T < 1) return 1;
  const int G = split_segments(N, T, H, kda_device_sms());
  return G > 1 && workspace_bytes >= split_seg_workspace_bytes(N, T, H, G) ? G : 1;
}

extern "C" kda_status kda_debug_split_segments(int segments) {
  g_force_segments.store(segments);
  return KDA_OK;
}

extern "C" kda_status kda_debug_stall_test(int flags) {
  if (flags < 0 || flags > 3) return KDA_ERR_INVALID_ARG;
  g_stall_test.store(flags);
  return KDA_OK;
}

// Test hook of the debug build (see kda.h): the record capacity the kernels
// are told; 0 restores the real one.
extern "C" kda_status kda_debug_record_capacity(int64_t items) {
  if (items < 0) return KDA_ERR_INVALID_ARG;
  g_record_capacity.store((long long)items);
  return KDA_OK;
}
