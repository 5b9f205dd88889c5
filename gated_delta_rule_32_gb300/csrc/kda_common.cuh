// kda_common.cuh -- definitions shared by the KDA kernels and the C ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// Device-side bounds checks of the debug build (-DKDA_DEBUG): a failed check
// records KDA_ERR_BOUNDS and skips the access instead of trapping.
#ifdef KDA_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// Floor on the per-step log-decay: each step keeps at least e^-5 ~ 0.67% of
// its state (Kimi K3 architecture, orkas.ai, "A lower bound that erased a
// GPU code path").
constexpr float kLogFloor = -5.0f;
// Tile length over which the bound holds the cumulative log-decay in
// [-80, 0] (same section).
constexpr int kTile = 16;

struct FwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* g;
  const void* beta;
  const float* init_state;
  void* out;
  float* final_state;
  const int32_t* cu_seqlens;  // device, may be null
  int32_t* dev_status;        // device, may be null
  // segments (dense batches only): sequence n is cut into nseg pieces of
  // seglen tokens (a multiple of 64) that run as independent chains
  int nseg;                   // 0 or 1: no segmentation
  int64_t seglen;
  const float* seg_init;      // [N][nseg][H][dk][dv] entry states of segments
  float* seg_final;           // [N][nseg][H][dk][dv] zero-start final states
  float* seg_P;               // [N][nseg][H][dk][dk] cumulative transitions
  float* ckpt;                // device, may be null: state checkpoints
  int ckpt_every;             // tokens between checkpoints (multiple of 64)
  int ckpt_max;               // checkpoint slots per (sequence, head)
  int N;                      // number of sequences
  int T;                      // tokens per batch row (packed: total)
  int H, dk, dv;
  float scale;
};

// a = max(-softplus(x), -5), softplus in its overflow-free form
// max(x, 0) + log1p(exp(-|x|)) (Towards AI walkthrough, "Kimi Delta
// Attention (KDA)": negative-softplus decay map; floor as above).
__device__ __forceinline__ float log_decay(float x) {
  float sp = fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x)));
  return fmaxf(-sp, kLogFloor);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Resolve the token span of sequence n.  Dense: row n, [0, T).  Packed:
// row 0, [cu[n], cu[n+1]).  Returns false (and records the error) when the
// packed offsets are malformed, so that no access leaves the buffers.
__device__ __forceinline__ bool seq_span(const FwdParams& p, int n, int64_t& row_base,
                                         int64_t& t0, int64_t& t1) {
  if (p.cu_seqlens == nullptr) {
    row_base = (int64_t)n * p.T;
    t0 = 0;
    t1 = p.T;
    return true;
  }
  row_base = 0;
  int32_t a = p.cu_seqlens[n];
  int32_t b = p.cu_seqlens[n + 1];
  bool ok = (a >= 0) && (b >= a) && (b <= p.T) && (n != 0 || a == 0) &&
            (n != p.N - 1 || b == p.T);
  if (!ok) {
    if (p.dev_status) atomicExch(p.dev_status, (int32_t)KDA_ERR_BAD_SEQLENS);
    return false;
  }
  t0 = a;
  t1 = b;
  return true;
}

}  // namespace kda

// Per-device launch set-up, kept per (device, kernel) for the life of the
// process and safe to call from several host threads at once (kda_api.cu).
// kda_smem_attr raises kernel `func`'s dynamic shared-memory limit to
// `bytes` on the current device, the first time that pair is seen;
// kda_device_sms returns the current device's SM count (0 if the runtime
// cannot tell).
kda_status kda_smem_attr(const void* func, int bytes);
int kda_device_sms();

// The argument rules of the C ABI (kda_api.cu): sizes, NULL pointers,
// alignment, the supported dk / dv / chunk / dtype, and no overlap of the
// output (or of a final state other than the initial one) with any input.
kda_status kda_check_args(const void* q, const void* k, const void* v, const void* g,
                          const void* beta, const float* s0, const void* out, const float* s1,
                          int B, int T, int H, int dk, int dv, const int32_t* cu, int dtype,
                          int chunk_size, int algo);

// Launchers (one per translation unit).
kda_status kda_launch_simt(const kda::FwdParams& p, kda_dtype dtype, cudaStream_t stream);
kda_status kda_launch_tc(const kda::FwdParams& p, cudaStream_t stream);
kda_status kda_launch_tc_summary(const kda::FwdParams& p, cudaStream_t stream);
kda_status kda_launch_seg_scan(const kda::FwdParams& p, cudaStream_t stream);
bool kda_tc_supported(int dk, int dv);
