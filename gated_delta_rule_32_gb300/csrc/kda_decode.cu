// kda_decode.cu -- the recurrent form for a few tokens per sequence: the
// decode step of serving, and the speculative-decoding rebuild (replaying
// the accepted tokens' cached projected inputs from a saved state, since an
// in-place state cannot be rolled back: Kimi K3 architecture, orkas.ai,
// "The cost is paid in the serving stack").
//
// Per token, for every (sequence, head), with S the dk x dv state:
//   S' = Diag(alpha) S;  p = S'^T k;  S = S' + beta k (v - p)^T;  o = S^T q
// One CTA per (sequence, head, 32 value channels); the CTA's 128 x 32 slice
// of S stays in registers (warp w owns key rows 16w .. 16w+15, lane j owns
// value channel j), so the state is read from and written to HBM once per
// call whatever the number of tokens.
#include "kda_common.cuh"

namespace {

constexpr int DC = 32;    // value channels per CTA
constexpr int NTD = 256;  // threads: 8 warps x 16 key rows = 128 key channels

template <typename Tin>
__global__ void __launch_bounds__(NTD) kda_decode_kernel(kda::FwdParams p) {
  __shared__ float s_a[128], s_k[128], s_q[128], s_v[DC], s_part[8][DC], s_pv[DC];
  __shared__ float s_beta;
  const int h = blockIdx.x, n = blockIdx.y, c0 = blockIdx.z * DC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, dk = p.dk, dv = p.dv;
  const int rows = dk / 8;  // key rows per warp (dk = 128 -> 16)
  const Tin* q = static_cast<const Tin*>(p.q);
  const Tin* k = static_cast<const Tin*>(p.k);
  const Tin* v = static_cast<const Tin*>(p.v);
  const Tin* g = static_cast<const Tin*>(p.g);
  const Tin* beta = static_cast<const Tin*>(p.beta);
  Tin* out = static_cast<Tin*>(p.out);

  float S[16];
  const int64_t sbase = ((int64_t)n * H + h) * (int64_t)dk * dv;
  const bool col_ok = lane < DC && c0 + lane < dv;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const int i = warp * rows + e;
    S[e] = (e < rows && col_ok && p.init_state) ? p.init_state[sbase + (int64_t)i * dv + c0 + lane]
                                                : 0.0f;
  }
  for (int t = 0; t < p.T; ++t) {
    const int64_t tok = ((int64_t)n * p.T + t) * H + h;
    if (tid < dk) {
      s_a[tid] = expf(kda::log_decay(kda::to_f32(g[tok * dk + tid])));
      s_k[tid] = kda::to_f32(k[tok * dk + tid]);
      s_q[tid] = kda::to_f32(q[tok * dk + tid]) * p.scale;
    } else if (tid < dk + DC) {
      const int j = tid - dk;
      s_v[j] = (c0 + j < dv) ? kda::to_f32(v[tok * dv + c0 + j]) : 0.0f;
    } else if (tid == dk + DC) {
      s_beta = kda::to_f32(beta[tok]);
    }
    __syncthreads();
    // S' = Diag(alpha) S and this warp's share of p = S'^T k
    float part = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      if (e < rows) {
        const int i = warp * rows + e;
        S[e] *= s_a[i];
        part = fmaf(s_k[i], S[e], part);
      }
    }
    s_part[warp][lane] = part;
    __syncthreads();
    if (warp == 0) {
      float pj = 0.0f;
#pragma unroll
      for (int w = 0; w < 8; ++w) pj += s_part[w][lane];
      s_pv[lane] = s_beta * (s_v[lane] - pj);  // beta (v - p)
    }
    __syncthreads();
    // S += k (beta (v - p))^T and this warp's share of o = S^T q
    const float bd = s_pv[lane];
    float op = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      if (e < rows) {
        const int i = warp * rows + e;
        S[e] = fmaf(s_k[i], bd, S[e]);
        op = fmaf(s_q[i], S[e], op);
      }
    }
    s_part[warp][lane] = op;
    __syncthreads();
    if (warp == 0 && col_ok) {
      float o = 0.0f;
#pragma unroll
      for (int w = 0; w < 8; ++w) o += s_part[w][lane];
      out[tok * dv + c0 + lane] = kda::from_f32<Tin>(o);
    }
    // the next token's loads overwrite s_a/s_k/s_q/s_v only after this point
    __syncthreads();
  }
  if (p.final_state && col_ok) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int i = warp * rows + e;
      if (e < rows) p.final_state[sbase + (int64_t)i * dv + c0 + lane] = S[e];
    }
  }
}

}  // namespace

extern "C" kda_status kda_decode(const void* q, const void* k, const void* v, const void* g_logit,
                                 const void* beta, float* state, void* out, int N, int T, int H,
                                 int dk, int dv, kda_dtype dtype, float scale,
                                 kda_stream_t stream) {
  if (!state || N < 1 || H < 1 || T < 0) return KDA_ERR_INVALID_ARG;
  if (T > 0 && (!q || !k || !v || !g_logit || !beta || !out)) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
  if (!(dk == 16 || dk == 32 || dk == 64 || dk == 128)) return KDA_ERR_UNSUPPORTED;
  if (!(dv == 16 || dv == 32 || dv == 64 || dv == 128)) return KDA_ERR_UNSUPPORTED;
  if (((uintptr_t)state & 15) != 0) return KDA_ERR_MISALIGNED;
  if (N > 65535 || H > 65535) return KDA_ERR_UNSUPPORTED;
  kda::FwdParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g_logit; p.beta = beta;
  p.init_state = state; p.final_state = state; p.out = out;
  p.N = N; p.T = T; p.H = H; p.dk = dk; p.dv = dv; p.scale = scale;
  dim3 grid(H, N, (dv + DC - 1) / DC);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == KDA_F32)
    kda_decode_kernel<float><<<grid, NTD, 0, s>>>(p);
  else
    kda_decode_kernel<__nv_bfloat16><<<grid, NTD, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
