// kda_simt.cu -- chunked KDA forward on the CUDA cores, fp32 arithmetic.
//
// The fp32 path (fp32 inputs need 1e-4 relative accuracy, beyond a BF16
// tensor-core product) and the fallback-free reference shape of the
// algorithm for every (dk, dv).  One CTA per (sequence, head, dv slice);
// the chunk is one 16-token tile, so the reference point of the decay
// factorisation is the chunk start and every factor stays in range:
//   Qh_r = q_r * e^{G_r}      in [e^-80, 1]      (G_r: cumulative log-decay
//   Kh_r = k_r * e^{G_r}                          from the chunk start)
//   Kt_i = k_i * e^{-G_i}     at most e^80
//   Kd_i = k_i * e^{G_C - G_i}
// (the 16-token bound of Kimi K3 architecture, orkas.ai, "A lower bound
// that erased a GPU code path").  Per chunk:
//   A_qk = tril(Qh Kt^T), A_kk = diag(beta) strict_tril(Kh Kt^T)
//   Tm = (I + A_kk)^{-1};  W = Tm diag(beta) Kh;  U = Tm diag(beta) V
//   Delta = U - W S;  O = Qh S + A_qk Delta;  S <- e^{G_C} * S + Kd^T Delta
// which is the recurrence S_t = (I - b k k^T) Diag(alpha) S + b k v^T,
// o_t = S_t^T q_t unrolled over the chunk (derivation in the oracle's chunk
// mirror).  Rows past the end of a sequence are padded with q = k = v = 0,
// beta = 0, log-decay 0.
#include "kda_common.cuh"

namespace {

constexpr int C = kda::kTile;   // chunk length of this path
constexpr int NT = 256;         // threads per CTA

template <int DK, int DVS>
struct SimtSmem {
  float Qh[C][DK + 1];
  float Kh[C][DK + 1];
  float Kt[C][DK + 1];
  float Kd[C][DK + 1];
  float W[C][DK + 1];
  float V[C][DVS];
  float U[C][DVS];
  float D[C][DVS];   // Delta
  float P[C][DVS];   // Qh S
  float Aqk[C][C + 1];
  float Akk[C][C + 1];
  float Tm[C][C + 1];
  float b[C];
  float gC[DK];      // e^{G_C}
  float S[DK][DVS];
};

template <int DK, int DVS, typename Tin>
__global__ void __launch_bounds__(NT) kda_simt_kernel(kda::FwdParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<SimtSmem<DK, DVS>*>(smem_raw);
  const int h = blockIdx.x, n = blockIdx.y, c0 = blockIdx.z * DVS;
  const int tid = threadIdx.x;
  const int H = p.H, dv = p.dv;

  int64_t row_base, t0, t1;
  if (!kda::seq_span(p, n, row_base, t0, t1)) return;

  const Tin* __restrict__ q = static_cast<const Tin*>(p.q);
  const Tin* __restrict__ k = static_cast<const Tin*>(p.k);
  const Tin* __restrict__ v = static_cast<const Tin*>(p.v);
  const Tin* __restrict__ g = static_cast<const Tin*>(p.g);
  const Tin* __restrict__ beta = static_cast<const Tin*>(p.beta);
  Tin* __restrict__ out = static_cast<Tin*>(p.out);

  const int64_t sbase = ((int64_t)n * H + h) * (int64_t)DK * dv;
  for (int idx = tid; idx < DK * DVS; idx += NT) {
    int i = idx / DVS, j = idx % DVS;
    sm.S[i][j] = p.init_state ? p.init_state[sbase + (int64_t)i * dv + c0 + j] : 0.0f;
  }

  for (int64_t cs = t0; cs < t1; cs += C) {
    const int L = (t1 - cs) < C ? (int)(t1 - cs) : C;
    __syncthreads();  // previous chunk fully consumed
    // ---- gate, cumulative log-decay, scaled operands -------------------
    if (tid < DK) {
      const int j = tid;
      float G[C];
      float acc = 0.0f;
#pragma unroll
      for (int r = 0; r < C; ++r) {
        float a = 0.0f;
        if (r < L) {
          int64_t tok = (row_base + cs + r) * H + h;
          a = kda::log_decay(kda::to_f32(g[tok * DK + j]));
        }
        acc += a;
        G[r] = acc;
      }
      const float GC = acc;
      sm.gC[j] = expf(GC);
#pragma unroll
      for (int r = 0; r < C; ++r) {
        float qv = 0.0f, kv = 0.0f;
        if (r < L) {
          int64_t tok = (row_base + cs + r) * H + h;
          qv = kda::to_f32(q[tok * DK + j]) * p.scale;
          kv = kda::to_f32(k[tok * DK + j]);
        }
        const float e = expf(G[r]);
        sm.Qh[r][j] = qv * e;
        sm.Kh[r][j] = kv * e;
        sm.Kt[r][j] = kv * expf(-G[r]);
        sm.Kd[r][j] = kv * expf(GC - G[r]);
      }
    }
    for (int idx = tid; idx < C * DVS; idx += NT) {
      int r = idx / DVS, c = idx % DVS;
      float x = 0.0f;
      if (r < L) x = kda::to_f32(v[((row_base + cs + r) * H + h) * dv + c0 + c]);
      sm.V[r][c] = x;
    }
    if (tid < C) {
      float x = 0.0f;
      if (tid < L) x = kda::to_f32(beta[(row_base + cs + tid) * H + h]);
      sm.b[tid] = x;
    }
    __syncthreads();
    // ---- Gram matrices: 136 A_qk entries (i <= r), 120 A_kk (i < r) ---------
    for (int e = tid; e < C * C; e += NT) {
      int r = e / C, i = e % C;
      float aq = 0.0f, ak = 0.0f;
      if (i <= r) {
        for (int j = 0; j < DK; ++j) {
          float kt = sm.Kt[i][j];
          aq = fmaf(sm.Qh[r][j], kt, aq);
          ak = fmaf(sm.Kh[r][j], kt, ak);
        }
      }
      sm.Aqk[r][i] = aq;
      sm.Akk[r][i] = (i < r) ? sm.b[r] * ak : 0.0f;
    }
    __syncthreads();
    // ---- Tm = (I + A_kk)^{-1}: lane c owns column c ------------------------
    if (tid < C) {
      const int c = tid;
      float col[C];
#pragma unroll
      for (int r = 0; r < C; ++r) {
        float x = (r == c) ? 1.0f : 0.0f;
        if (r > c) {
#pragma unroll
          for (int i = 0; i < r; ++i) x = fmaf(-sm.Akk[r][i], col[i], x);
        }
        col[r] = x;
      }
#pragma unroll
      for (int r = 0; r < C; ++r) sm.Tm[r][c] = col[r];
    }
    __syncthreads();
    // ---- W = Tm diag(b) Kh, U = Tm diag(b) V ------------------------------
    for (int idx = tid; idx < C * DK; idx += NT) {
      int r = idx / DK, j = idx % DK;
      float acc = 0.0f;
      for (int i = 0; i <= r; ++i) acc = fmaf(sm.Tm[r][i] * sm.b[i], sm.Kh[i][j], acc);
      sm.W[r][j] = acc;
    }
    for (int idx = tid; idx < C * DVS; idx += NT) {
      int r = idx / DVS, c = idx % DVS;
      float acc = 0.0f;
      for (int i = 0; i <= r; ++i) acc = fmaf(sm.Tm[r][i] * sm.b[i], sm.V[i][c], acc);
      sm.U[r][c] = acc;
    }
    __syncthreads();
    // ---- Delta = U - W S, P = Qh S ----------------------------------------
    for (int idx = tid; idx < C * DVS; idx += NT) {
      int r = idx / DVS, c = idx % DVS;
      float ws = 0.0f, qs = 0.0f;
      for (int j = 0; j < DK; ++j) {
        float s = sm.S[j][c];
        ws = fmaf(sm.W[r][j], s, ws);
        qs = fmaf(sm.Qh[r][j], s, qs);
      }
      sm.D[r][c] = sm.U[r][c] - ws;
      sm.P[r][c] = qs;
    }
    __syncthreads();
    // ---- O = P + A_qk Delta; S <- e^{G_C} S + Kd^T Delta ------------------
    for (int idx = tid; idx < C * DVS; idx += NT) {
      int r = idx / DVS, c = idx % DVS;
      float acc = sm.P[r][c];
      for (int i = 0; i <= r; ++i) acc = fmaf(sm.Aqk[r][i], sm.D[i][c], acc);
      if (r < L) out[((row_base + cs + r) * H + h) * dv + c0 + c] = kda::from_f32<Tin>(acc);
    }
    for (int idx = tid; idx < DK * DVS; idx += NT) {
      int j = idx / DVS, c = idx % DVS;
      float acc = sm.gC[j] * sm.S[j][c];
#pragma unroll
      for (int r = 0; r < C; ++r) acc = fmaf(sm.Kd[r][j], sm.D[r][c], acc);
      sm.S[j][c] = acc;
      // state checkpoint after every `ckpt_every` tokens of the sequence
      if (p.ckpt) {
        const int64_t done = cs + L - t0;
        if (L == C && done % p.ckpt_every == 0) {
          const int64_t slot = done / p.ckpt_every - 1;
          if (slot < p.ckpt_max)
            p.ckpt[((((int64_t)n * H + h) * p.ckpt_max + slot) * DK + j) * dv + c0 + c] = acc;
        }
      }
    }
  }
  __syncthreads();
  if (p.final_state) {
    for (int idx = tid; idx < DK * DVS; idx += NT) {
      int i = idx / DVS, j = idx % DVS;
      p.final_state[sbase + (int64_t)i * dv + c0 + j] = sm.S[i][j];
    }
  }
}

template <int DK, int DVS, typename Tin>
kda_status launch(const kda::FwdParams& p, cudaStream_t stream) {
  const size_t smem = sizeof(SimtSmem<DK, DVS>);
  auto kern = kda_simt_kernel<DK, DVS, Tin>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return KDA_ERR_CUDA;
  dim3 grid(p.H, p.N, p.dv / DVS);
  kern<<<grid, NT, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

template <typename Tin>
kda_status dispatch(const kda::FwdParams& p, cudaStream_t stream) {
  // dv slice per CTA: all of dv up to 64 columns
#define KDA_SIMT_CASE(DK_)                                            \
  if (p.dk == DK_) {                                                  \
    if (p.dv >= 64) return launch<DK_, 64, Tin>(p, stream);           \
    if (p.dv == 32) return launch<DK_, 32, Tin>(p, stream);           \
    return launch<DK_, 16, Tin>(p, stream);                           \
  }
  KDA_SIMT_CASE(16)
  KDA_SIMT_CASE(32)
  KDA_SIMT_CASE(64)
  KDA_SIMT_CASE(128)
#undef KDA_SIMT_CASE
  return KDA_ERR_UNSUPPORTED;
}

}  // namespace

kda_status kda_launch_simt(const kda::FwdParams& p, kda_dtype dtype, cudaStream_t stream) {
  if (dtype == KDA_F32) return dispatch<float>(p, stream);
  return dispatch<__nv_bfloat16>(p, stream);
}
