// kda_decode.cu -- the recurrent form for a few tokens per sequence: the
// decode step of serving, and the speculative-decoding rebuild (replaying
// the accepted tokens' cached projected inputs from a saved state, since an
// in-place state cannot be rolled back: Kimi K3 architecture, orkas.ai,
// "The cost is paid in the serving stack").
//
// Per token, for every (sequence, head), with S the dk x dv state:
//   S' = Diag(alpha) S;  p = S'^T k;  S = S' + beta k (v - p)^T;  o = S^T q
// One CTA per (sequence, head, 128 value channels): warp w owns value
// channels 16w .. 16w+15 and lane l channel 16w + (l mod 16) over half the
// key rows (lanes 0-15 the first half, 16-31 the second), its part of the
// column of S in registers.  So the state is read from and written to HBM
// once per call whatever the number of tokens, in 64-byte row segments, and
// the two sums over the key rows of every token (p and o) take one shuffle
// each: no barrier per token.  The CTA stages the inputs of up to TB tokens
// at a time (the decays taken for all of them at once) and the warps then
// run their tokens independently.
#include "kda_common.cuh"

namespace {

constexpr int NTD = 256;  // threads: 8 warps x 16 value channels
constexpr int DCB = 128;  // value channels per CTA
constexpr int TB = 16;    // tokens staged in shared memory at a time

template <typename Tin, int DK>
__global__ void __launch_bounds__(NTD, 2) kda_decode_kernel(kda::FwdParams p) {
  constexpr int RH = DK / 2;  // key rows per lane
  __shared__ __align__(16) float s_a[TB][DK], s_k[TB][DK], s_q[TB][DK];
  __shared__ float s_v[TB][DCB], s_beta[TB];
  const int h = blockIdx.x, n = blockIdx.y, c0 = blockIdx.z * DCB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, dv = p.dv;
  const int jl = 16 * warp + (lane & 15);  // value channel within the CTA
  const int j = c0 + jl;
  const int r0 = (lane >> 4) * RH;         // this lane's first key row
  const bool col_ok = j < dv;
  const Tin* q = static_cast<const Tin*>(p.q);
  const Tin* k = static_cast<const Tin*>(p.k);
  const Tin* v = static_cast<const Tin*>(p.v);
  const Tin* g = static_cast<const Tin*>(p.g);
  const Tin* beta = static_cast<const Tin*>(p.beta);
  Tin* out = static_cast<Tin*>(p.out);

  const int64_t sbase = ((int64_t)n * H + h) * (int64_t)DK * dv;
  float S[RH];
#pragma unroll
  for (int i = 0; i < RH; ++i)
    S[i] = (col_ok && p.init_state) ? p.init_state[sbase + (int64_t)(r0 + i) * dv + j] : 0.0f;
  for (int t0 = 0; t0 < p.T; t0 += TB) {
    const int nt = p.T - t0 < TB ? p.T - t0 : TB;
    auto tok_of = [&](int tt) { return ((int64_t)n * p.T + t0 + tt) * H + h; };
    for (int e = tid; e < nt * DK; e += NTD) {
      const int tt = e / DK, i = e - tt * DK;
      const int64_t tok = tok_of(tt);
      s_a[tt][i] = expf(kda::log_decay(kda::to_f32(g[tok * DK + i])));
      s_k[tt][i] = kda::to_f32(k[tok * DK + i]);
      s_q[tt][i] = kda::to_f32(q[tok * DK + i]) * p.scale;
    }
    for (int e = tid; e < nt * DCB; e += NTD) {
      const int tt = e / DCB, c = e - tt * DCB;
      s_v[tt][c] = (c0 + c < dv) ? kda::to_f32(v[tok_of(tt) * dv + c0 + c]) : 0.0f;
    }
    if (tid < nt) s_beta[tid] = kda::to_f32(beta[tok_of(tid)]);
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      // S' = Diag(alpha) S, p = S'^T k (this lane's rows, then the other half)
      float pa = 0.0f, pb = 0.0f;
#pragma unroll
      for (int i = 0; i < RH; i += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(&s_a[tt][r0 + i]);
        const float4 k4 = *reinterpret_cast<const float4*>(&s_k[tt][r0 + i]);
        S[i] *= a4.x; S[i + 1] *= a4.y; S[i + 2] *= a4.z; S[i + 3] *= a4.w;
        pa = fmaf(k4.x, S[i], pa);
        pb = fmaf(k4.y, S[i + 1], pb);
        pa = fmaf(k4.z, S[i + 2], pa);
        pb = fmaf(k4.w, S[i + 3], pb);
      }
      float pp = pa + pb;
      pp += __shfl_xor_sync(0xffffffffu, pp, 16);
      // S += k (beta (v - p)), o = S^T q
      const float d = s_beta[tt] * (s_v[tt][jl] - pp);
      float oa = 0.0f, ob = 0.0f;
#pragma unroll
      for (int i = 0; i < RH; i += 4) {
        const float4 k4 = *reinterpret_cast<const float4*>(&s_k[tt][r0 + i]);
        const float4 q4 = *reinterpret_cast<const float4*>(&s_q[tt][r0 + i]);
        S[i] = fmaf(k4.x, d, S[i]);
        S[i + 1] = fmaf(k4.y, d, S[i + 1]);
        S[i + 2] = fmaf(k4.z, d, S[i + 2]);
        S[i + 3] = fmaf(k4.w, d, S[i + 3]);
        oa = fmaf(q4.x, S[i], oa);
        ob = fmaf(q4.y, S[i + 1], ob);
        oa = fmaf(q4.z, S[i + 2], oa);
        ob = fmaf(q4.w, S[i + 3], ob);
      }
      float o = oa + ob;
      o += __shfl_xor_sync(0xffffffffu, o, 16);
      if (col_ok && lane < 16) out[tok_of(tt) * dv + j] = kda::from_f32<Tin>(o);
    }
    // the next block's staging overwrites the inputs only after this point
    __syncthreads();
  }
  if (p.final_state && col_ok) {
#pragma unroll
    for (int i = 0; i < RH; ++i) p.final_state[sbase + (int64_t)(r0 + i) * dv + j] = S[i];
  }
}

template <typename Tin>
void launch_decode(const kda::FwdParams& p, dim3 grid, cudaStream_t s) {
  switch (p.dk) {
    case 16: kda_decode_kernel<Tin, 16><<<grid, NTD, 0, s>>>(p); break;
    case 32: kda_decode_kernel<Tin, 32><<<grid, NTD, 0, s>>>(p); break;
    case 64: kda_decode_kernel<Tin, 64><<<grid, NTD, 0, s>>>(p); break;
    default: kda_decode_kernel<Tin, 128><<<grid, NTD, 0, s>>>(p); break;
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
  dim3 grid(H, N, (dv + DCB - 1) / DCB);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == KDA_F32)
    launch_decode<float>(p, grid, s);
  else
    launch_decode<__nv_bfloat16>(p, grid, s);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
