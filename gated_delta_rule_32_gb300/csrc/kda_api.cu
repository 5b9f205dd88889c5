// kda_api.cu -- the C ABI of libkda.so: argument checks, path selection,
// the end-to-end host-buffer call.  Every step of the forward runs in the
// library's own kernels; there is no CPU fallback.
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "kda_common.cuh"

namespace {
std::mutex g_dev_mu;
std::map<std::pair<int, const void*>, int> g_smem_set;  // (device, kernel) -> bytes set
std::map<int, int> g_sms;                                // device -> SM count
}  // namespace

kda_status kda_smem_attr(const void* func, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  auto key = std::make_pair(dev, func);
  auto it = g_smem_set.find(key);
  if (it != g_smem_set.end() && it->second >= bytes) return KDA_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return KDA_ERR_CUDA;
  g_smem_set[key] = bytes;
  return KDA_OK;
}

int kda_device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  auto it = g_sms.find(dev);
  if (it != g_sms.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 0;
  g_sms[dev] = n;
  return n;
}

size_t kda_split_packed_workspace_bytes(int N, int T, int H);
size_t kda_split_packed_min_workspace_bytes(int N, int T, int H);

namespace {

bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + nb && b0 < a0 + na;
}

struct Sizes {
  size_t qk, v, beta, state, cu;  // bytes
};

Sizes sizes_of(int B, int T, int H, int dk, int dv, int esz, int packed) {
  Sizes s;
  const size_t rows = packed ? 1 : (size_t)B;
  s.qk = rows * (size_t)T * H * dk * esz;
  s.v = rows * (size_t)T * H * dv * esz;
  s.beta = rows * (size_t)T * H * esz;
  s.state = (size_t)B * H * dk * dv * sizeof(float);
  s.cu = packed ? (size_t)(B + 1) * sizeof(int32_t) : 0;
  return s;
}

kda_status check_args(const void* q, const void* k, const void* v, const void* g,
                      const void* beta, const float* s0, const void* out, const float* s1,
                      int B, int T, int H, int dk, int dv, const int32_t* cu, int dtype,
                      int chunk_size, int algo) {
  if (B < 1 || T < 0 || H < 1) return KDA_ERR_INVALID_ARG;
  // with no tokens nothing is read or written but the states
  if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
  if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
  if (chunk_size != 0 && chunk_size != 16 && chunk_size != 64) return KDA_ERR_UNSUPPORTED;
  if (algo < KDA_ALGO_AUTO || algo > KDA_ALGO_SPLIT) return KDA_ERR_INVALID_ARG;
  const int esz = dtype == KDA_F32 ? 4 : 2;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) ||
      !aligned(out, 16) || !aligned(beta, esz))
    return KDA_ERR_MISALIGNED;
  if ((s0 && !aligned(s0, 16)) || (s1 && !aligned(s1, 16)) || (cu && !aligned(cu, 4)))
    return KDA_ERR_MISALIGNED;
  Sizes s = sizes_of(B, T, H, dk, dv, esz, cu != nullptr);
  if (overlap(out, s.v, q, s.qk) || overlap(out, s.v, k, s.qk) || overlap(out, s.v, g, s.qk) ||
      overlap(out, s.v, v, s.v) || overlap(out, s.v, beta, s.beta) ||
      overlap(out, s.v, s0, s.state) || overlap(out, s.v, s1, s.state))
    return KDA_ERR_INVALID_ARG;
  if (s1 && s0 != s1 &&
      (overlap(s1, s.state, q, s.qk) || overlap(s1, s.state, k, s.qk) ||
       overlap(s1, s.state, g, s.qk) || overlap(s1, s.state, v, s.v) ||
       overlap(s1, s.state, s0, s.state)))
    return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

int sm_count() {
  const int n = kda_device_sms();
  return n > 0 ? n : 148;
}

// Segments per sequence for the tensor-core path: only dense batches whose
// (sequence, head) chains would leave more than half of the SMs idle, with
// segments of at least 1024 tokens.
int auto_segments(int B, int T, int H, int sms) {
  const int ctas = B * H * 2;  // two CTAs (value halves) per chain
  if (ctas * 2 > sms || T < 2048) return 1;
  int nseg = sms / ctas;
  const int by_len = T / 1024;
  if (nseg > by_len) nseg = by_len;
  return nseg < 2 ? 1 : nseg;
}

bool use_tc(int dtype, int dk, int dv, int chunk_size, int algo) {
  if (algo == KDA_ALGO_SIMT) return false;
  if (dtype != KDA_BF16 || chunk_size == 16) return false;
  return kda_tc_supported(dk, dv);
}

// The two-kernel form of the tensor-core path, when asked for or by default
// (it runs every chunk's state-independent work at once; the fused kernel
// repeats it per value half and runs it serially per chain), dense or packed
// (long batches in slices of chunks or of chunk columns); KDA_ALGO_TC always
// takes the fused kernel.
bool use_split(int dtype, int dk, int dv, int chunk_size, int algo, int packed, int N, int T,
               int H) {
  (void)H;
  if (T < 1 || !use_tc(dtype, dk, dv, chunk_size, algo)) return false;
  if (algo != KDA_ALGO_SPLIT && algo != KDA_ALGO_AUTO) return false;
  if (packed && (N < 1 || N >= (1 << 24))) return false;
  return true;
}

}  // namespace

kda_status kda_check_args(const void* q, const void* k, const void* v, const void* g,
                          const void* beta, const float* s0, const void* out, const float* s1,
                          int B, int T, int H, int dk, int dv, const int32_t* cu, int dtype,
                          int chunk_size, int algo) {
  return check_args(q, k, v, g, beta, s0, out, s1, B, T, H, dk, dv, cu, dtype, chunk_size,
                    algo);
}

kda_status kda_run_segmented(const kda::FwdParams& p, int nseg, void* scratch,
                             cudaStream_t stream);
size_t kda_seg_scratch_bytes(int N, int H, int nseg, int dk, int dv);
kda_status kda_run_split(const kda::FwdParams& p, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);
size_t kda_split_workspace_bytes(int N, int T, int H);
size_t kda_split_min_workspace_bytes(int N, int H);
kda_status kda_run_split_range(const kda::FwdParams& p, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream, int c0, int cnt);
size_t kda_split_slice_workspace_bytes(int N, int H, int chunks);
kda_status kda_run_split_packed_range(const kda::FwdParams& p, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream, int g0,
                                      int cnt, bool prepare);
int kda_split_packed_g_max(int N, int T);
size_t kda_split_packed_slice_workspace_bytes(int N, int T, int H, int cols);

namespace {
// The end-to-end call on the two-kernel path runs the batch in pieces of
// whole chunks (a dense batch: chunks [c0, c1) of every sequence; a packed
// one: chunk columns [g0, g1), which are one contiguous range of token
// rows): the inputs of piece i + 1 go to the device on two copy streams
// while piece i runs on the caller's stream and the output of piece i - 1
// comes back on a third, so the host link, not the sum of copies and
// kernels, sets the time.  The state crosses pieces exactly as it crosses
// slices (fp32, unchanged), so the result does not depend on the cut.
constexpr int kHostPieces = 8;
int host_piece_chunks(int T) {
  const int nchunks = (T + 63) / 64;
  const int pieces = nchunks < kHostPieces ? nchunks : kHostPieces;
  return (nchunks + pieces - 1) / pieces;
}
// chunk columns per piece of a packed batch (of the bound ceil(T / 64) + N)
int host_piece_cols(int N, int T) {
  const int g = kda_split_packed_g_max(N, T);
  const int pieces = g < kHostPieces ? g : kHostPieces;
  return (g + pieces - 1) / pieces;
}
bool host_pipelined(int dtype, int dk, int dv, int packed, int N, int T) {
  if (packed)
    return use_split(dtype, dk, dv, 0, KDA_ALGO_AUTO, 1, N, T, 1) &&
           kda_split_packed_g_max(N, T) >= 2;
  return use_split(dtype, dk, dv, 0, KDA_ALGO_AUTO, 0, 1, T, 1) && (T + 63) / 64 >= 2;
}
size_t host_piece_workspace_bytes(int N, int T, int H, int packed) {
  return packed ? kda_split_packed_slice_workspace_bytes(N, T, H, host_piece_cols(N, T))
                : kda_split_slice_workspace_bytes(N, H, host_piece_chunks(T));
}
}  // namespace
// A workspace smaller than the default (but at least the minimum) runs the
// sequence in more, shorter slices.
static kda_status run_split_ws(const kda::FwdParams& p, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
  const bool packed = p.cu_seqlens != nullptr;
  if (workspace) {
    const size_t min_bytes = packed ? kda_split_packed_min_workspace_bytes(p.N, p.T, p.H)
                                    : kda_split_min_workspace_bytes(p.N, p.H);
    if (workspace_bytes < min_bytes) return KDA_ERR_WORKSPACE;
    return kda_run_split(p, workspace, workspace_bytes, stream);
  }
  const size_t need = packed ? kda_split_packed_workspace_bytes(p.N, p.T, p.H)
                             : kda_split_workspace_bytes(p.N, p.T, p.H);
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, need, stream) != cudaSuccess) return KDA_ERR_CUDA;
  kda_status st = kda_run_split(p, ws, need, stream);
  if (cudaFreeAsync(ws, stream) != cudaSuccess && st == KDA_OK) st = KDA_ERR_CUDA;
  return st;
}

static kda_status run_segmented_ws(const kda::FwdParams& p, int nseg, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream) {
  const size_t need = kda_seg_scratch_bytes(p.N, p.H, nseg, p.dk, p.dv);
  if (workspace) {
    if (workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 255) != 0) return KDA_ERR_MISALIGNED;
    return kda_run_segmented(p, nseg, workspace, stream);
  }
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, need, stream) != cudaSuccess) return KDA_ERR_CUDA;
  kda_status st = kda_run_segmented(p, nseg, ws, stream);
  if (cudaFreeAsync(ws, stream) != cudaSuccess && st == KDA_OK) st = KDA_ERR_CUDA;
  return st;
}

extern "C" {

const char* kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: null pointer, bad size or aliasing";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: dk/dv/chunk/dtype not supported";
    case KDA_ERR_MISALIGNED: return "KDA_ERR_MISALIGNED: pointer alignment rule broken";
    case KDA_ERR_BAD_SEQLENS: return "KDA_ERR_BAD_SEQLENS: cu_seqlens malformed";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: bounded on-chip wait gave up";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime error";
    case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace too small";
    case KDA_ERR_BOUNDS: return "KDA_ERR_BOUNDS: device-side bounds check failed (debug build)";
  }
  return "KDA_ERR_UNKNOWN";
}

const char* kda_build_info(void) {
#ifdef KDA_DEBUG
  return "libkda: KDA chunked forward, sm_103a (tcgen05/TMEM/TMA tensor-core paths + fp32 "
         "CUDA-core path), debug build with device-side bounds checks";
#else
  return "libkda: KDA chunked forward, sm_103a (tcgen05/TMEM/TMA tensor-core paths + fp32 "
         "CUDA-core path)";
#endif
}

int kda_resolve_algo(int dtype, int dk, int dv, int chunk_size, int algo) {
  if (dtype != KDA_BF16 && dtype != KDA_F32) return -1;
  if (!dim_ok(dk) || !dim_ok(dv)) return -1;
  if (chunk_size != 0 && chunk_size != 16 && chunk_size != 64) return -1;
  if (algo < KDA_ALGO_AUTO || algo > KDA_ALGO_SPLIT) return -1;
  const bool tc = use_tc(dtype, dk, dv, chunk_size, algo);
  if ((algo == KDA_ALGO_TC || algo == KDA_ALGO_SPLIT) && !tc) return -1;
  if (algo == KDA_ALGO_SPLIT) return KDA_ALGO_SPLIT;
  return tc ? KDA_ALGO_TC : KDA_ALGO_SIMT;
}

int kda_resolve_path(int N, int T, int H, int dk, int dv, int dtype, int chunk_size, int algo,
                     int packed) {
  const int fam = kda_resolve_algo(dtype, dk, dv, chunk_size, algo);
  if (fam < 0 || N < 1 || H < 1 || T < 0) return -1;
  if (fam == KDA_ALGO_SIMT) return KDA_ALGO_SIMT;
  if (algo == KDA_ALGO_TC) return KDA_ALGO_TC;
  if (!use_split(dtype, dk, dv, chunk_size, algo, packed, N, T, H)) return KDA_ALGO_TC;
  return KDA_ALGO_SPLIT;
}

size_t kda_workspace_bytes(int N, int T, int H, int dk, int dv, int dtype, int chunk_size,
                           int algo, int packed) {
  if (N < 1 || H < 1 || T < 1) return 0;
  if (!use_tc(dtype, dk, dv, chunk_size, algo)) return 0;
  if (use_split(dtype, dk, dv, chunk_size, algo, packed, N, T, H))
    return packed ? kda_split_packed_workspace_bytes(N, T, H) : kda_split_workspace_bytes(N, T, H);
  if (packed) return 0;
  const int nseg = auto_segments(N, T, H, sm_count());
  return nseg > 1 ? kda_seg_scratch_bytes(N, H, nseg, dk, dv) : 0;
}

static kda_status fwd_impl(const void* q, const void* k, const void* v, const void* g_logit,
                           const void* beta, const float* init_state, void* out,
                           float* final_state, int B, int T, int H, int dk, int dv,
                           const int32_t* cu_seqlens, kda_dtype dtype, int chunk_size,
                           float scale, int algo, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, float* ckpt, int ckpt_every, int ckpt_max,
                           kda_stream_t stream_);

kda_status kda_chunk_fwd_ex(const void* q, const void* k, const void* v, const void* g_logit,
                            const void* beta, const float* init_state, void* out,
                            float* final_state, int B, int T, int H, int dk, int dv,
                            const int32_t* cu_seqlens, kda_dtype dtype, int chunk_size,
                            float scale, int algo, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, kda_stream_t stream_) {
  return fwd_impl(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk, dv,
                  cu_seqlens, dtype, chunk_size, scale, algo, workspace, workspace_bytes,
                  dev_status, nullptr, 0, 0, stream_);
}

kda_status kda_chunk_fwd_ckpt(const void* q, const void* k, const void* v, const void* g_logit,
                              const void* beta, const float* init_state, void* out,
                              float* final_state, int B, int T, int H, int dk, int dv,
                              const int32_t* cu_seqlens, kda_dtype dtype, float scale,
                              float* checkpoints, int every, int max_per_seq,
                              int32_t* dev_status, kda_stream_t stream_) {
  if (!checkpoints || every <= 0 || every % 64 != 0 || max_per_seq < 1)
    return KDA_ERR_INVALID_ARG;
  if (!aligned(checkpoints, 16)) return KDA_ERR_MISALIGNED;
  return fwd_impl(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk, dv,
                  cu_seqlens, dtype, 0, scale, KDA_ALGO_AUTO, nullptr, 0, dev_status,
                  checkpoints, every, max_per_seq, stream_);
}

static kda_status fwd_impl(const void* q, const void* k, const void* v, const void* g_logit,
                           const void* beta, const float* init_state, void* out,
                           float* final_state, int B, int T, int H, int dk, int dv,
                           const int32_t* cu_seqlens, kda_dtype dtype, int chunk_size,
                           float scale, int algo, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, float* ckpt, int ckpt_every, int ckpt_max,
                           kda_stream_t stream_) {
  kda_status st = check_args(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk,
                             dv, cu_seqlens, dtype, chunk_size, algo);
  if (st != KDA_OK) return st;
  // (each path checks the size of a workspace it is given)
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  kda::FwdParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g_logit; p.beta = beta;
  p.init_state = init_state; p.out = out; p.final_state = final_state;
  p.cu_seqlens = cu_seqlens; p.dev_status = dev_status;
  p.N = B; p.T = T; p.H = H; p.dk = dk; p.dv = dv; p.scale = scale;
  p.ckpt = ckpt; p.ckpt_every = ckpt_every; p.ckpt_max = ckpt_max;
  if ((algo == KDA_ALGO_TC || algo == KDA_ALGO_SPLIT) && !use_tc(dtype, dk, dv, chunk_size, algo))
    return KDA_ERR_UNSUPPORTED;
  if (!use_tc(dtype, dk, dv, chunk_size, algo)) return kda_launch_simt(p, dtype, stream);
  if (use_split(dtype, dk, dv, chunk_size, algo, cu_seqlens != nullptr, B, T, H))
    return run_split_ws(p, workspace, workspace_bytes, stream);
  if (algo == KDA_ALGO_SPLIT) return KDA_ERR_UNSUPPORTED;
  const int nseg = (cu_seqlens || ckpt) ? 1 : auto_segments(B, T, H, sm_count());
  if (nseg <= 1) return kda_launch_tc(p, stream);
  return run_segmented_ws(p, nseg, workspace, workspace_bytes, stream);
}

kda_status kda_chunk_fwd_seg(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                             const uint16_t* g_logit, const uint16_t* beta,
                             const float* init_state, uint16_t* out, float* final_state, int B,
                             int T, int H, int dk, int dv, float scale, int nseg,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status,
                             kda_stream_t stream_) {
  kda_status st = check_args(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk,
                             dv, nullptr, KDA_BF16, 0, KDA_ALGO_TC);
  if (st != KDA_OK) return st;
  if (!kda_tc_supported(dk, dv)) return KDA_ERR_UNSUPPORTED;
  if (nseg < 1 || nseg > 4096) return KDA_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  kda::FwdParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g_logit; p.beta = beta;
  p.init_state = init_state; p.out = out; p.final_state = final_state;
  p.dev_status = dev_status;
  p.N = B; p.T = T; p.H = H; p.dk = dk; p.dv = dv; p.scale = scale;
  if (nseg == 1 || T == 0) return kda_launch_tc(p, stream);
  return run_segmented_ws(p, nseg, workspace, workspace_bytes, stream);
}

size_t kda_seg_workspace_bytes(int B, int H, int nseg, int dk, int dv) {
  if (B < 1 || H < 1 || nseg < 2) return 0;
  return kda_seg_scratch_bytes(B, H, nseg, dk, dv);
}

kda_status kda_chunk_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const uint16_t* g_logit, const uint16_t* beta,
                         const float* init_state, uint16_t* out, float* final_state,
                         int B, int T, int H, int dk, int dv, const int32_t* cu_seqlens,
                         kda_stream_t stream) {
  return kda_chunk_fwd_ex(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk,
                          dv, cu_seqlens, KDA_BF16, 0, 1.0f, KDA_ALGO_AUTO, nullptr, 0,
                          nullptr, stream);
}

kda_status kda_chunk_fwd_f32(const float* q, const float* k, const float* v,
                             const float* g_logit, const float* beta,
                             const float* init_state, float* out, float* final_state,
                             int B, int T, int H, int dk, int dv, const int32_t* cu_seqlens,
                             kda_stream_t stream) {
  return kda_chunk_fwd_ex(q, k, v, g_logit, beta, init_state, out, final_state, B, T, H, dk,
                          dv, cu_seqlens, KDA_F32, 0, 1.0f, KDA_ALGO_AUTO, nullptr, 0,
                          nullptr, stream);
}

static size_t round_up(size_t x) { return (x + 255) & ~(size_t)255; }

size_t kda_host_staging_bytes(int B, int T, int H, int dk, int dv, int dtype, int has_init,
                              int has_final, int packed) {
  if (B < 1 || T < 0 || H < 1 || dk < 1 || dv < 1) return 0;
  const int esz = dtype == KDA_F32 ? 4 : 2;
  Sizes s = sizes_of(B, T, H, dk, dv, esz, packed);
  size_t tot = 3 * round_up(s.qk) + 2 * round_up(s.v) + round_up(s.beta);
  if (has_init) tot += round_up(s.state);
  if (has_final) tot += round_up(s.state);
  tot += round_up(s.cu) + 256;  // cu_seqlens + device status word
  // the path's own workspace (chunk records of one piece of the two-kernel
  // form, or the segment scratch), so that the end-to-end call allocates
  // nothing itself
  if (host_pipelined(dtype, dk, dv, packed, B, T))
    tot += round_up(host_piece_workspace_bytes(B, T, H, packed));
  else
    tot += round_up(kda_workspace_bytes(B, T, H, dk, dv, dtype, 0, KDA_ALGO_AUTO, packed));
  return tot;
}

}  // extern "C"

namespace {
// The pieces of a pipelined end-to-end call (see host_piece_chunks): bf16,
// dk = dv = 128, dense.  Returns once everything is back on the host.
kda_status host_pipelined_run(const void* q, const void* k, const void* v, const void* g_logit,
                              const void* beta, const float* init_state, void* out,
                              float* final_state, int B, int T, int H, float scale, char* dq,
                              char* dk_, char* dv_, char* dg, char* db, float* ds0, char* dout,
                              float* ds1, int32_t* dstat, void* ws, size_t ws_bytes,
                              cudaStream_t stream) {
  constexpr int D = 128;
  const size_t row_qk = (size_t)H * D * 2, row_b = (size_t)H * 2;  // bytes per token row
  const int nchunks = (T + 63) / 64, per = host_piece_chunks(T);
  const int pieces = (nchunks + per - 1) / per;
  cudaStream_t s_in[2] = {nullptr, nullptr}, s_out = nullptr;
  cudaEvent_t ev0 = nullptr, ev_in[2][kHostPieces] = {}, ev_c[kHostPieces] = {};
  kda_status st = KDA_OK;
  auto cu = [&](cudaError_t e) {
    if (e != cudaSuccess && st == KDA_OK) st = KDA_ERR_CUDA;
    return st == KDA_OK;
  };
  cu(cudaStreamCreateWithFlags(&s_in[0], cudaStreamNonBlocking));
  cu(cudaStreamCreateWithFlags(&s_in[1], cudaStreamNonBlocking));
  cu(cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking));
  cu(cudaEventCreateWithFlags(&ev0, cudaEventDisableTiming));
  for (int i = 0; i < pieces; ++i) {
    cu(cudaEventCreateWithFlags(&ev_in[0][i], cudaEventDisableTiming));
    cu(cudaEventCreateWithFlags(&ev_in[1][i], cudaEventDisableTiming));
    cu(cudaEventCreateWithFlags(&ev_c[i], cudaEventDisableTiming));
  }
  int32_t hstat = 0;
  if (st == KDA_OK) {
    kda::FwdParams p{};
    p.q = dq; p.k = dk_; p.v = dv_; p.g = dg; p.beta = db;
    p.init_state = ds0; p.out = dout; p.final_state = ds1; p.dev_status = dstat;
    p.N = B; p.T = T; p.H = H; p.dk = D; p.dv = D; p.scale = scale;
    // the copies start after whatever the caller queued on its stream
    cu(cudaMemsetAsync(dstat, 0, sizeof(int32_t), stream));
    cu(cudaEventRecord(ev0, stream));
    cu(cudaStreamWaitEvent(s_in[0], ev0, 0));
    cu(cudaStreamWaitEvent(s_in[1], ev0, 0));
    auto h2d = [&](char* dst, const void* src, size_t off, size_t n, cudaStream_t sm) {
      return cu(cudaMemcpyAsync(dst + off, static_cast<const char*>(src) + off, n,
                                cudaMemcpyHostToDevice, sm));
    };
    for (int i = 0; i < pieces && st == KDA_OK; ++i) {
      const int c0 = i * per, cnt = nchunks - c0 < per ? nchunks - c0 : per;
      const size_t t0 = (size_t)c0 * 64;
      const size_t t1 = (size_t)(c0 + cnt) * 64 < (size_t)T ? (size_t)(c0 + cnt) * 64 : (size_t)T;
      for (int n = 0; n < B; ++n) {  // rows [t0, t1) of each sequence
        const size_t r0 = (size_t)n * T + t0, nr = t1 - t0;
        h2d(dq, q, r0 * row_qk, nr * row_qk, s_in[0]);
        h2d(dk_, k, r0 * row_qk, nr * row_qk, s_in[0]);
        h2d(dg, g_logit, r0 * row_qk, nr * row_qk, s_in[1]);
        h2d(dv_, v, r0 * row_qk, nr * row_qk, s_in[1]);
        h2d(db, beta, r0 * row_b, nr * row_b, s_in[1]);
      }
      if (i == 0 && ds0)
        h2d(reinterpret_cast<char*>(ds0), init_state, 0, (size_t)B * H * D * D * 4, s_in[0]);
      cu(cudaEventRecord(ev_in[0][i], s_in[0]));
      cu(cudaEventRecord(ev_in[1][i], s_in[1]));
      cu(cudaStreamWaitEvent(stream, ev_in[0][i], 0));
      cu(cudaStreamWaitEvent(stream, ev_in[1][i], 0));
      if (st == KDA_OK) st = kda_run_split_range(p, ws, ws_bytes, stream, c0, cnt);
      cu(cudaEventRecord(ev_c[i], stream));
      cu(cudaStreamWaitEvent(s_out, ev_c[i], 0));
      for (int n = 0; n < B; ++n) {
        const size_t off = ((size_t)n * T + t0) * row_qk;
        cu(cudaMemcpyAsync(static_cast<char*>(out) + off, dout + off, (t1 - t0) * row_qk,
                           cudaMemcpyDeviceToHost, s_out));
      }
    }
    if (ds1)
      cu(cudaMemcpyAsync(final_state, ds1, (size_t)B * H * D * D * 4, cudaMemcpyDeviceToHost,
                         s_out));
    cu(cudaMemcpyAsync(&hstat, dstat, sizeof(int32_t), cudaMemcpyDeviceToHost, s_out));
  }
  // everything queued is waited for, whatever failed
  for (cudaStream_t sm : {s_in[0], s_in[1], s_out, stream})
    if (sm || sm == stream) cu(cudaStreamSynchronize(sm));
  for (int i = 0; i < pieces; ++i) {
    if (ev_in[0][i]) cudaEventDestroy(ev_in[0][i]);
    if (ev_in[1][i]) cudaEventDestroy(ev_in[1][i]);
    if (ev_c[i]) cudaEventDestroy(ev_c[i]);
  }
  if (ev0) cudaEventDestroy(ev0);
  for (cudaStream_t sm : {s_in[0], s_in[1], s_out})
    if (sm) cudaStreamDestroy(sm);
  if (st == KDA_OK && hstat != 0) st = (kda_status)hstat;
  return st;
}

// The pieces of a pipelined end-to-end call on a packed batch: chunk columns
// [g0, g0 + per) of the bound ceil(T / 64) + N, each a contiguous range of
// token rows [row(g0), row(g0 + per)).  A piece's kernels also read up to 63
// rows past its range (the tile of a sequence's last, short chunk; those
// rows enter with zero weight), so each piece's copy reaches 64 rows
// further, and every row is copied once.  cu_seqlens: host offsets, already
// checked.
kda_status host_pipelined_packed_run(const void* q, const void* k, const void* v,
                                     const void* g_logit, const void* beta,
                                     const float* init_state, void* out, float* final_state,
                                     int N, int T, int H, float scale, const int32_t* cu,
                                     char* dq, char* dk_, char* dv_, char* dg, char* db,
                                     float* ds0, char* dout, float* ds1, int32_t* dcu,
                                     int32_t* dstat, void* ws, size_t ws_bytes,
                                     cudaStream_t stream) {
  constexpr int D = 128;
  const size_t row_qk = (size_t)H * D * 2, row_b = (size_t)H * 2;  // bytes per token row
  // first column of each sequence (ceil(len / 64) columns each)
  std::vector<int64_t> off(N + 1, 0);
  for (int n = 0; n < N; ++n) off[n + 1] = off[n] + (cu[n + 1] - cu[n] + 63) / 64;
  const int64_t cols = off[N];
  auto row_of = [&](int64_t g) -> int64_t {  // first token row of column g
    if (g >= cols) return T;
    const int n = (int)(std::upper_bound(off.begin(), off.end(), g) - off.begin()) - 1;
    return cu[n] + 64 * (g - off[n]);
  };
  const int g_max = kda_split_packed_g_max(N, T), per = host_piece_cols(N, T);
  const int pieces = (g_max + per - 1) / per;
  cudaStream_t s_in[2] = {nullptr, nullptr}, s_out = nullptr;
  cudaEvent_t ev0 = nullptr, ev_in[2][kHostPieces] = {}, ev_c[kHostPieces] = {};
  kda_status st = KDA_OK;
  auto cu_ok = [&](cudaError_t e) {
    if (e != cudaSuccess && st == KDA_OK) st = KDA_ERR_CUDA;
    return st == KDA_OK;
  };
  cu_ok(cudaStreamCreateWithFlags(&s_in[0], cudaStreamNonBlocking));
  cu_ok(cudaStreamCreateWithFlags(&s_in[1], cudaStreamNonBlocking));
  cu_ok(cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking));
  cu_ok(cudaEventCreateWithFlags(&ev0, cudaEventDisableTiming));
  for (int i = 0; i < pieces; ++i) {
    cu_ok(cudaEventCreateWithFlags(&ev_in[0][i], cudaEventDisableTiming));
    cu_ok(cudaEventCreateWithFlags(&ev_in[1][i], cudaEventDisableTiming));
    cu_ok(cudaEventCreateWithFlags(&ev_c[i], cudaEventDisableTiming));
  }
  int32_t hstat = 0;
  if (st == KDA_OK) {
    kda::FwdParams p{};
    p.q = dq; p.k = dk_; p.v = dv_; p.g = dg; p.beta = db;
    p.init_state = ds0; p.out = dout; p.final_state = ds1; p.dev_status = dstat;
    p.cu_seqlens = dcu;
    p.N = N; p.T = T; p.H = H; p.dk = D; p.dv = D; p.scale = scale;
    // the offsets and status word on the caller's stream, ahead of the
    // first piece's chunk table
    cu_ok(cudaMemcpyAsync(dcu, cu, (size_t)(N + 1) * sizeof(int32_t), cudaMemcpyHostToDevice,
                          stream));
    cu_ok(cudaMemsetAsync(dstat, 0, sizeof(int32_t), stream));
    cu_ok(cudaEventRecord(ev0, stream));
    cu_ok(cudaStreamWaitEvent(s_in[0], ev0, 0));
    cu_ok(cudaStreamWaitEvent(s_in[1], ev0, 0));
    auto h2d = [&](char* dst, const void* src, size_t off_b, size_t n, cudaStream_t sm) {
      return cu_ok(cudaMemcpyAsync(dst + off_b, static_cast<const char*>(src) + off_b, n,
                                   cudaMemcpyHostToDevice, sm));
    };
    int64_t copied = 0;  // rows [0, copied) are on the device or queued
    for (int i = 0; i < pieces && st == KDA_OK; ++i) {
      const int g0 = i * per, cnt = g_max - g0 < per ? g_max - g0 : per;
      const int64_t r0 = row_of(g0), r1 = row_of((int64_t)g0 + cnt);
      const int64_t need = r1 + 64 < T ? r1 + 64 : T;
      if (need > copied) {
        const size_t a = (size_t)copied, nr = (size_t)(need - copied);
        h2d(dq, q, a * row_qk, nr * row_qk, s_in[0]);
        h2d(dk_, k, a * row_qk, nr * row_qk, s_in[0]);
        h2d(dg, g_logit, a * row_qk, nr * row_qk, s_in[1]);
        h2d(dv_, v, a * row_qk, nr * row_qk, s_in[1]);
        h2d(db, beta, a * row_b, nr * row_b, s_in[1]);
        copied = need;
      }
      if (i == 0 && ds0)
        h2d(reinterpret_cast<char*>(ds0), init_state, 0, (size_t)N * H * D * D * 4, s_in[0]);
      cu_ok(cudaEventRecord(ev_in[0][i], s_in[0]));
      cu_ok(cudaEventRecord(ev_in[1][i], s_in[1]));
      cu_ok(cudaStreamWaitEvent(stream, ev_in[0][i], 0));
      cu_ok(cudaStreamWaitEvent(stream, ev_in[1][i], 0));
      if (st == KDA_OK) st = kda_run_split_packed_range(p, ws, ws_bytes, stream, g0, cnt, i == 0);
      cu_ok(cudaEventRecord(ev_c[i], stream));
      cu_ok(cudaStreamWaitEvent(s_out, ev_c[i], 0));
      if (r1 > r0)
        cu_ok(cudaMemcpyAsync(static_cast<char*>(out) + (size_t)r0 * row_qk,
                              dout + (size_t)r0 * row_qk, (size_t)(r1 - r0) * row_qk,
                              cudaMemcpyDeviceToHost, s_out));
    }
    if (ds1)
      cu_ok(cudaMemcpyAsync(final_state, ds1, (size_t)N * H * D * D * 4, cudaMemcpyDeviceToHost,
                            s_out));
    cu_ok(cudaMemcpyAsync(&hstat, dstat, sizeof(int32_t), cudaMemcpyDeviceToHost, s_out));
  }
  // everything queued is waited for, whatever failed
  for (cudaStream_t sm : {s_in[0], s_in[1], s_out, stream})
    if (sm || sm == stream) cu_ok(cudaStreamSynchronize(sm));
  for (int i = 0; i < pieces; ++i) {
    if (ev_in[0][i]) cudaEventDestroy(ev_in[0][i]);
    if (ev_in[1][i]) cudaEventDestroy(ev_in[1][i]);
    if (ev_c[i]) cudaEventDestroy(ev_c[i]);
  }
  if (ev0) cudaEventDestroy(ev0);
  for (cudaStream_t sm : {s_in[0], s_in[1], s_out})
    if (sm) cudaStreamDestroy(sm);
  if (st == KDA_OK && hstat != 0) st = (kda_status)hstat;
  return st;
}
}  // namespace

extern "C" {

kda_status kda_chunk_fwd_host(const void* q, const void* k, const void* v, const void* g_logit,
                              const void* beta, const float* init_state, void* out,
                              float* final_state, int B, int T, int H, int dk, int dv,
                              const int32_t* cu_seqlens, kda_dtype dtype, float scale,
                              void* dev_buffer, size_t dev_buffer_bytes, kda_stream_t stream_) {
  if (B < 1 || T < 0 || H < 1) return KDA_ERR_INVALID_ARG;
  if (T > 0 && (!q || !k || !v || !g_logit || !beta || !out)) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
  if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const int packed = cu_seqlens != nullptr;
  if (packed) {  // host-visible offsets: check them before any copy
    if (cu_seqlens[0] != 0 || cu_seqlens[B] != T) return KDA_ERR_BAD_SEQLENS;
    for (int n = 0; n < B; ++n)
      if (cu_seqlens[n + 1] < cu_seqlens[n]) return KDA_ERR_BAD_SEQLENS;
  }
  const int esz = dtype == KDA_F32 ? 4 : 2;
  Sizes s = sizes_of(B, T, H, dk, dv, esz, packed);
  const size_t need = kda_host_staging_bytes(B, T, H, dk, dv, dtype, init_state != nullptr,
                                             final_state != nullptr, packed);
  char* base = static_cast<char*>(dev_buffer);
  bool owned = false;
  if (!base) {
    if (cudaMallocAsync((void**)&base, need, stream) != cudaSuccess) return KDA_ERR_CUDA;
    owned = true;
  } else if (dev_buffer_bytes < need) {
    return KDA_ERR_WORKSPACE;
  }
  size_t off = 0;
  auto take = [&](size_t n) { char* p = base + off; off += round_up(n); return p; };
  char *dq = take(s.qk), *dk_ = take(s.qk), *dg = take(s.qk), *dv_ = take(s.v),
       *dout = take(s.v), *db = take(s.beta);
  float* ds0 = init_state ? (float*)take(s.state) : nullptr;
  float* ds1 = final_state ? (float*)take(s.state) : nullptr;
  int32_t* dcu = packed ? (int32_t*)take(s.cu) : nullptr;
  int32_t* dstat = (int32_t*)take(sizeof(int32_t));
  const bool piped = host_pipelined(dtype, dk, dv, packed, B, T);
  const size_t ws_bytes =
      piped ? host_piece_workspace_bytes(B, T, H, packed)
            : kda_workspace_bytes(B, T, H, dk, dv, dtype, 0, KDA_ALGO_AUTO, packed);
  void* ws = ws_bytes ? take(ws_bytes) : nullptr;
  if (piped) {
    kda_status st =
        packed ? host_pipelined_packed_run(q, k, v, g_logit, beta, init_state, out, final_state,
                                           B, T, H, scale, cu_seqlens, dq, dk_, dv_, dg, db, ds0,
                                           dout, ds1, dcu, dstat, ws, ws_bytes, stream)
               : host_pipelined_run(q, k, v, g_logit, beta, init_state, out, final_state, B, T,
                                    H, scale, dq, dk_, dv_, dg, db, ds0, dout, ds1, dstat, ws,
                                    ws_bytes, stream);
    if (owned) cudaFreeAsync(base, stream);
    if (cudaStreamSynchronize(stream) != cudaSuccess && st == KDA_OK) st = KDA_ERR_CUDA;
    return st;
  }
  kda_status st = KDA_OK;
  int32_t hstat = 0;
  bool ok = true;
  ok = ok && cudaMemcpyAsync(dq, q, s.qk, cudaMemcpyHostToDevice, stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(dk_, k, s.qk, cudaMemcpyHostToDevice, stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(dg, g_logit, s.qk, cudaMemcpyHostToDevice, stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(dv_, v, s.v, cudaMemcpyHostToDevice, stream) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(db, beta, s.beta, cudaMemcpyHostToDevice, stream) == cudaSuccess;
  if (ds0)
    ok = ok &&
         cudaMemcpyAsync(ds0, init_state, s.state, cudaMemcpyHostToDevice, stream) == cudaSuccess;
  if (dcu)
    ok = ok && cudaMemcpyAsync(dcu, cu_seqlens, s.cu, cudaMemcpyHostToDevice, stream) ==
                   cudaSuccess;
  if (!ok) st = KDA_ERR_CUDA;
  if (st == KDA_OK)
    st = kda_chunk_fwd_ex(dq, dk_, dv_, dg, db, ds0, dout, ds1, B, T, H, dk, dv, dcu, dtype, 0,
                          scale, KDA_ALGO_AUTO, ws, ws_bytes, dstat, stream_);
  if (st == KDA_OK) {
    ok = cudaMemcpyAsync(out, dout, s.v, cudaMemcpyDeviceToHost, stream) == cudaSuccess;
    if (ds1)
      ok = ok && cudaMemcpyAsync(final_state, ds1, s.state, cudaMemcpyDeviceToHost, stream) ==
                     cudaSuccess;
    ok = ok &&
         cudaMemcpyAsync(&hstat, dstat, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) ==
             cudaSuccess;
    if (!ok) st = KDA_ERR_CUDA;
  }
  if (owned) cudaFreeAsync(base, stream);
  if (cudaStreamSynchronize(stream) != cudaSuccess && st == KDA_OK) st = KDA_ERR_CUDA;
  if (st == KDA_OK && hstat != 0) st = (kda_status)hstat;
  return st;
}

}  // extern "C"
