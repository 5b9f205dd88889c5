// kda_cp.cu -- the pieces of context parallelism that run on a GPU.
//
// The state update of a span of tokens is affine in the state entering it:
// running the span from S_in gives S_out = P S_in + S0, where P (dk x dk) is
// the span's cumulative transition and S0 its final state from a zero start
// (Kimi K3 architecture, orkas.ai, "The cost is paid in the serving stack";
// Towards AI walkthrough, "Infrastructure co-design": a cumulative transition
// and a zero-initialised state per device, then a prefix scan and one
// fixed-size all-gather).  When the token axis of a batch is split across
// devices, device r computes the (P, S0) of its span (kda_segment_summary),
// the summaries of all devices are all-gathered (fixed size), and device r
// folds those of the devices before it into its entry state
// (kda_state_compose) before running its span.  The exchange itself belongs
// to the caller (torch.distributed in the package's Python layer).
#include "kda_common.cuh"

namespace {

constexpr int DK = 128, DV = 128;
constexpr int SC = 32;        // value columns per CTA
constexpr int LDP = DK + 1;   // padded row of P in shared memory

// S = P_{m-1} ( ... (P_0 S_init + S0_0) ... ) + S0_{m-1} for one (sequence,
// head) and 32 value columns; summaries[j] holds [P block | S0 block] with
// P [N][H][DK][DK] then S0 [N][H][DK][DV].  grid (H, N, DV / 32), 256
// threads: thread = (key row i, 16 columns).
__global__ void __launch_bounds__(256) kda_compose_kernel(const float* summaries, int m,
                                                          const float* init_state, float* out,
                                                          int N, int H) {
  extern __shared__ float sm[];
  float* sP = sm;               // [DK][LDP]
  float* sS = sP + DK * LDP;    // [DK][SC]
  const int h = blockIdx.x, n = blockIdx.y, c0 = blockIdx.z * SC;
  const int tid = threadIdx.x, i = tid & (DK - 1), cg = (tid >> 7) * 16;
  const int64_t nh = (int64_t)n * H + h;
  const int64_t p_block = (int64_t)N * H * DK * DK;
  const int64_t stride = p_block + (int64_t)N * H * DK * DV;
  for (int e = tid; e < DK * SC; e += 256) {
    const int r = e / SC, c = e % SC;
    sS[e] = init_state ? init_state[(nh * DK + r) * DV + c0 + c] : 0.0f;
  }
  for (int j = 0; j < m; ++j) {
    const float* P = summaries + j * stride + nh * DK * DK;
    const float* S0 = summaries + j * stride + p_block + nh * DK * DV;
    __syncthreads();
    for (int e = tid; e < DK * DK; e += 256) sP[(e / DK) * LDP + (e % DK)] = P[e];
    __syncthreads();
    float acc[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] = S0[(int64_t)i * DV + c0 + cg + c];
    for (int k = 0; k < DK; ++k) {
      const float pv = sP[i * LDP + k];
#pragma unroll
      for (int c = 0; c < 16; ++c) acc[c] = fmaf(pv, sS[k * SC + cg + c], acc[c]);
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 16; ++c) sS[i * SC + cg + c] = acc[c];
  }
  __syncthreads();
  for (int e = tid; e < DK * SC; e += 256) {
    const int r = e / SC, c = e % SC;
    out[(nh * DK + r) * DV + c0 + c] = sS[e];
  }
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

}  // namespace

extern "C" size_t kda_summary_floats(int N, int H, int dk, int dv) {
  if (N < 1 || H < 1 || dk < 1 || dv < 1) return 0;
  return (size_t)N * H * ((size_t)dk * dk + (size_t)dk * dv);
}

extern "C" kda_status kda_segment_summary(const uint16_t* q, const uint16_t* k,
                                          const uint16_t* v, const uint16_t* g_logit,
                                          const uint16_t* beta, float* summary, int B, int T,
                                          int H, int dk, int dv, int32_t* dev_status,
                                          kda_stream_t stream_) {
  if (B < 1 || T < 0 || H < 1 || !summary) return KDA_ERR_INVALID_ARG;
  if (T > 0 && (!q || !k || !v || !g_logit || !beta)) return KDA_ERR_INVALID_ARG;
  if (!kda_tc_supported(dk, dv)) return KDA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g_logit) ||
      !aligned16(summary) || ((uintptr_t)beta & 1) != 0)
    return KDA_ERR_MISALIGNED;
  // the summary must not overlap any input
  const size_t sb = kda_summary_floats(B, H, dk, dv) * sizeof(float);
  const size_t qb = (size_t)B * T * H * dk * 2, bb = (size_t)B * T * H * 2;
  auto over = [&](const void* a, size_t na) {
    if (!a || na == 0) return false;
    const uintptr_t a0 = (uintptr_t)a, s0 = (uintptr_t)summary;
    return a0 < s0 + sb && s0 < a0 + na;
  };
  if (over(q, qb) || over(k, qb) || over(v, qb) || over(g_logit, qb) || over(beta, bb))
    return KDA_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  kda::FwdParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g_logit; p.beta = beta;
  p.dev_status = dev_status;
  p.N = B; p.T = T; p.H = H; p.dk = dk; p.dv = dv; p.scale = 1.0f;
  // one segment per sequence: the whole span [0, T)
  p.nseg = 1;
  p.seglen = T;
  p.seg_P = summary;
  p.seg_final = summary + (size_t)B * H * dk * dk;
  return kda_launch_tc_summary(p, stream);
}

extern "C" kda_status kda_state_compose(const float* summaries, int m, const float* init_state,
                                        float* state_out, int N, int H, int dk, int dv,
                                        kda_stream_t stream_) {
  if (m < 0 || N < 1 || H < 1 || !state_out || (m > 0 && !summaries))
    return KDA_ERR_INVALID_ARG;
  if (dk != DK || dv != DV) return KDA_ERR_UNSUPPORTED;
  if (N > 65535 || H > 65535) return KDA_ERR_UNSUPPORTED;
  if (!aligned16(state_out) || (init_state && !aligned16(init_state)) ||
      (summaries && !aligned16(summaries)))
    return KDA_ERR_MISALIGNED;
  const size_t smem = sizeof(float) * (DK * LDP + DK * SC);
  if (kda_smem_attr((const void*)kda_compose_kernel, (int)smem) != KDA_OK) return KDA_ERR_CUDA;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  kda_compose_kernel<<<dim3(H, N, DV / SC), 256, smem, stream>>>(summaries, m, init_state,
                                                                  state_out, N, H);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
