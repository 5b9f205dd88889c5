// kda_seg_static.cu -- the segment-parallel forward for callers that cannot
// allocate device memory.
//
// Some callers run where no allocation may happen: a serving engine that has
// already reserved all of the GPU's memory for its own pools (state caches,
// weights) and forbids any further cudaMalloc/cudaMallocAsync at request
// time, or a host framework that calls this library as an extension and
// neither hands it a workspace nor lets it allocate one.  For them this
// entry point keeps the segment scratch in a fixed array compiled into the
// library, so a call allocates nothing.
#include <mutex>

#include "kda_common.cuh"

kda_status kda_run_segmented(const kda::FwdParams& p, int nseg, void* scratch,
                             cudaStream_t stream);
size_t kda_seg_scratch_bytes(int N, int H, int nseg, int dk, int dv);

namespace {

// 16 MiB: room for N * H * nseg <= 85 (sequence, head, segment) triples at
// dk = dv = 128 (192 KiB each), e.g. 16 heads of one sequence in 5 segments.
constexpr size_t kStaticScratchBytes = (size_t)16 << 20;
__device__ __align__(256) unsigned char kda_seg_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the array on the current device, looked up once per
// device (the host-side symbol is only a stand-in, never a device address).
kda_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, kda_seg_static_scratch) != cudaSuccess || !ptr)
      return KDA_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_seg_static(const uint16_t* q, const uint16_t* k,
                                               const uint16_t* v, const uint16_t* g_logit,
                                               const uint16_t* beta, const float* init_state,
                                               uint16_t* out, float* final_state, int B, int T,
                                               int H, int dk, int dv, float scale, int nseg,
                                               int32_t* dev_status, kda_stream_t stream_) {
  // the same argument rules as kda_chunk_fwd_seg
  kda_status st = kda_check_args(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H,
                                 dk, dv, nullptr, KDA_BF16, 0, KDA_ALGO_TC);
  if (st != KDA_OK) return st;
  if (!kda_tc_supported(dk, dv)) return KDA_ERR_UNSUPPORTED;
  if (nseg < 2 || nseg > 4096) return KDA_ERR_INVALID_ARG;
  // everything beyond the fixed array is refused before anything is queued
  if (kda_seg_scratch_bytes(B, H, nseg, dk, dv) > kStaticScratchBytes) return KDA_ERR_WORKSPACE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  kda::FwdParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g_logit; p.beta = beta;
  p.init_state = init_state; p.out = out; p.final_state = final_state;
  p.dev_status = dev_status;
  p.N = B; p.T = T; p.H = H; p.dk = dk; p.dv = dv; p.scale = scale;
  if (T == 0) {  // no tokens: the states pass through, as in kda_chunk_fwd_seg
    if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), stream) != cudaSuccess)
      return KDA_ERR_CUDA;
    return kda_launch_tc(p, stream);
  }
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != KDA_OK) return st;
  if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  return kda_run_segmented(p, nseg, scratch, stream);
}
