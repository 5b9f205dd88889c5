// kda_seg.cu -- segment-parallel forward for long sequences with few
// (sequence, head) chains.
//
// The state update of a segment is affine in its entry state: running the
// segment from S_in gives S_out = P S_in + S0, where P (dk x dk) is the
// segment's cumulative transition and S0 its final state from a zero start
// (the decomposition into a cumulative transition and a zero-initialised
// state: Kimi K3 architecture, orkas.ai, "The cost is paid in the serving
// stack"; Towards AI walkthrough, "Infrastructure co-design").  So:
//   pass 1 (every segment in parallel): P and S0 of each segment, no output
//           (the fused kernel in its summary mode);
//   pass 2 (serial over segments, tiny): S_in(s) = P(s-1) S_in(s-1) + S0(s-1);
//   pass 3 (every segment in parallel): the fused forward of each segment
//           from its resolved entry state, writing the output.
// The scratch holds S0, P and S_in of every (sequence, segment, head).
#include "kda_common.cuh"

namespace {

constexpr int DK = 128;
constexpr int SC = 32;         // value columns per scan CTA
constexpr int LDP = DK + 1;    // padded row of P in shared memory

// pass 2: grid (H, N, dv / 32), 256 threads; thread = (key row i, 16 columns)
__global__ void __launch_bounds__(256) kda_seg_scan_kernel(kda::FwdParams p) {
  extern __shared__ float sm[];
  float* sP = sm;                 // [DK][LDP]
  float* sS = sP + DK * LDP;      // [DK][SC] entry state of the previous segment
  const int h = blockIdx.x, n = blockIdx.y, c0 = blockIdx.z * SC;
  const int tid = threadIdx.x, i = tid & (DK - 1), cg = (tid >> 7) * 16;
  const int H = p.H, dv = p.dv, nseg = p.nseg;
  for (int e = tid; e < DK * SC; e += 256) {
    const int r = e / SC, c = e % SC;
    sS[e] = p.init_state ? p.init_state[(((int64_t)n * H + h) * DK + r) * dv + c0 + c] : 0.0f;
  }
  for (int s = 1; s < nseg; ++s) {
    const int64_t prev = ((int64_t)n * nseg + (s - 1)) * H + h;
    const float* P = p.seg_P + prev * DK * DK;
    __syncthreads();
    for (int e = tid; e < DK * DK; e += 256) sP[(e / DK) * LDP + (e % DK)] = P[e];
    __syncthreads();
    float acc[16];
    const float* S0 = p.seg_final + prev * DK * dv + (int64_t)i * dv + c0 + cg;
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] = S0[c];
    for (int k = 0; k < DK; ++k) {
      const float pv = sP[i * LDP + k];
#pragma unroll
      for (int c = 0; c < 16; ++c) acc[c] = fmaf(pv, sS[k * SC + cg + c], acc[c]);
    }
    __syncthreads();
    float* dst = const_cast<float*>(p.seg_init) +
                 (((int64_t)n * nseg + s) * H + h) * DK * dv + (int64_t)i * dv + c0 + cg;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      sS[i * SC + cg + c] = acc[c];
      dst[c] = acc[c];
    }
  }
}

}  // namespace

kda_status kda_launch_seg_scan(const kda::FwdParams& p, cudaStream_t stream) {
  const size_t smem = sizeof(float) * (DK * LDP + DK * SC);
  if (kda_smem_attr((const void*)kda_seg_scan_kernel, (int)smem) != KDA_OK) return KDA_ERR_CUDA;
  dim3 grid(p.H, p.N, p.dv / SC);
  kda_seg_scan_kernel<<<grid, 256, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// Bytes of segment scratch for N sequences, H heads, nseg segments.
size_t kda_seg_scratch_bytes(int N, int H, int nseg, int dk, int dv) {
  const size_t per = (size_t)N * nseg * H;
  return per * ((size_t)2 * dk * dv + (size_t)dk * dk) * sizeof(float);
}

// The three passes over a dense bf16 batch; `scratch` holds at least
// kda_seg_scratch_bytes() bytes (256-byte aligned).
kda_status kda_run_segmented(const kda::FwdParams& p0, int nseg, void* scratch,
                             cudaStream_t stream) {
  kda::FwdParams p = p0;
  const size_t per = (size_t)p.N * nseg * p.H;
  float* base = static_cast<float*>(scratch);
  p.nseg = nseg;
  p.seglen = (((int64_t)p.T + nseg - 1) / nseg + 63) / 64 * 64;
  p.seg_final = base;
  p.seg_init = base + per * p.dk * p.dv;
  p.seg_P = base + 2 * per * p.dk * p.dv;
  kda::FwdParams p1 = p;          // pass 1: summaries, no output, no checkpoints
  p1.final_state = nullptr;
  p1.ckpt = nullptr;
  kda_status st = kda_launch_tc_summary(p1, stream);
  if (st != KDA_OK) return st;
  st = kda_launch_seg_scan(p, stream);
  if (st != KDA_OK) return st;
  p.ckpt = nullptr;               // checkpoints are a property of the whole sequence
  return kda_launch_tc(p, stream);
}
