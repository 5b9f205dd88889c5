// kda_probe.cu -- a single-tile tcgen05 GEMM used by the tests to check the
// operand layouts and descriptors the fused kernel relies on: D = A * B^T
// for one M x N x K tile, A and B given row-major (K contiguous) in global
// memory, staged by the CTA into shared memory (K-major or MN-major core
// matrices) or, for A, into tensor memory.  The raw accumulator (all 128
// TMEM lanes x N columns) is returned so the tests can also read the lane
// placement of an M = 64 tile.  Not on the forward path.
#include "kda_common.cuh"
#include "sm100.cuh"

namespace {

constexpr int kProbeThreads = 128;
constexpr uint32_t kSentinel = 0x7fc00001u;  // a quiet NaN marks untouched lanes

struct ProbeArgs {
  const uint16_t* A;  // [M][K]
  const uint16_t* B;  // [N][K]
  float* D;           // [128][N]
  int32_t* status;
  int M, N, K;
  int a_mode;  // 0 smem K-major, 1 smem MN-major, 2 tmem
  int b_mode;  // 0 smem K-major, 1 smem MN-major, 2 smem MN-major 128-byte swizzle (N = 64)
  int pack;    // 0: core matrices adjacent along K first; 1: along M/N first
};

// byte offset of element (r, k) of an R x K operand, and its (lbo, sbo)
__device__ __forceinline__ uint32_t op_off(int r, int k, int R, int K, int mn_major, int pack,
                                           uint32_t& lbo, uint32_t& sbo) {
  if (!mn_major) {
    if (pack == 0) { lbo = 128; sbo = (uint32_t)(K / 8) * 128; }
    else { sbo = 128; lbo = (uint32_t)(R / 8) * 128; }
    return (r / 8) * sbo + (k / 8) * lbo + (r % 8) * 16 + (k % 8) * 2;
  }
  if (pack == 0) { sbo = 128; lbo = (uint32_t)(R / 8) * 128; }
  else { lbo = 128; sbo = (uint32_t)(K / 8) * 128; }
  return (r / 8) * sbo + (k / 8) * lbo + (k % 8) * 16 + (r % 8) * 2;
}

__global__ void __launch_bounds__(kProbeThreads) umma_probe_kernel(ProbeArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid / 32;
  unsigned char* sA = smem;                 // 32 KiB
  unsigned char* sB = smem + 32768;         // 64 KiB (+ slack after)
  // a swizzled operand starts on a 1024-byte boundary (its atoms' alignment)
  sB += (1024u - (sm100::smem_u32(sB) & 1023u)) & 1023u;
  const int M = a.M, N = a.N, K = a.K;

  if (warp == 0) {
    sm100::tmem_alloc(&tmem_base, 512);
    sm100::tmem_relinquish();
  }
  if (tid == 0) {
    sm100::mbar_init(&bar, 1);
    sm100::fence_mbar_init();
  }
  uint32_t lbo_a = 0, sbo_a = 0, lbo_b = 0, sbo_b = 0;
  for (int e = tid; e < M * K; e += kProbeThreads) {
    int r = e / K, k = e % K;
    uint32_t o = op_off(r, k, M, K, a.a_mode == 1, a.pack, lbo_a, sbo_a);
    if (a.a_mode != 2) *reinterpret_cast<uint16_t*>(sA + o) = a.A[e];
  }
  op_off(0, 0, M, K, a.a_mode == 1, a.pack, lbo_a, sbo_a);
  for (int e = tid; e < N * K; e += kProbeThreads) {
    int r = e / K, k = e % K;
    uint32_t o;
    if (a.b_mode == 2) {
      // element (n, k): atom k / 8, row k % 8 of it (128 bytes), 16-byte chunk
      // n / 8 stored at chunk (n / 8) ^ (k % 8)
      o = (uint32_t)(k >> 3) * 1024u + (uint32_t)(k & 7) * 128u +
          ((uint32_t)(((r >> 3) ^ (k & 7)) & 7) << 4) + (uint32_t)(r & 7) * 2u;
    } else {
      o = op_off(r, k, N, K, a.b_mode == 1, a.pack, lbo_b, sbo_b);
    }
    *reinterpret_cast<uint16_t*>(sB + o) = a.B[e];
  }
  if (a.b_mode == 2) {
    lbo_b = 1024; sbo_b = 1024;  // one atom along N: only the K-atom stride matters
  } else {
    op_off(0, 0, N, K, a.b_mode == 1, a.pack, lbo_b, sbo_b);
  }
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t d_col = 0, a_col = 256;  // D in columns [0, N), A in [256, 256 + K/2)
  const uint32_t lane0 = 32u * (warp % 4);
  // sentinel over the whole D region; A rows (lane = row) when A is in TMEM
  for (int c = 0; c < N; c += 16) {
    uint32_t r[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = kSentinel;
    sm100::tmem_st16(sm100::taddr(tbase, lane0, d_col + c), r);
  }
  if (a.a_mode == 2) {
    const int row = lane0 + (tid % 32);
    for (int c = 0; c < K / 2; c += 16) {
      uint32_t r[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        int k = 2 * (c + i);
        uint32_t lo = 0, hi = 0;
        if (row < M) { lo = a.A[row * K + k]; hi = a.A[row * K + k + 1]; }
        r[i] = lo | (hi << 16);
      }
      sm100::tmem_st16(sm100::taddr(tbase, lane0, a_col + c), r);
    }
  }
  sm100::tmem_wait_st();
  sm100::fence_async_smem();
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  if (tid == 0) {
    const uint32_t idesc = sm100::idesc_bf16(M, N, a.a_mode == 1, a.b_mode != 0);
    for (int s = 0; s < K / 16; ++s) {
      uint64_t bd = a.b_mode == 2
                        ? sm100::smem_desc_sw128(sm100::smem_u32(sB) + s * 2048, lbo_b, sbo_b)
                        : sm100::smem_desc(sm100::smem_u32(sB) + s * 2 * lbo_b, lbo_b, sbo_b);
      if (a.a_mode == 2) {
        sm100::mma_ts(tbase + d_col, tbase + a_col + 8 * s, bd, idesc, s > 0);
      } else {
        uint64_t ad = sm100::smem_desc(sm100::smem_u32(sA) + s * 2 * lbo_a, lbo_a, sbo_a);
        sm100::mma_ss(tbase + d_col, ad, bd, idesc, s > 0);
      }
    }
    sm100::mma_commit(&bar);
  }
  __syncwarp();
  const bool ok = sm100::mbar_wait(&bar, 0);
  if (!ok && a.status) atomicExch(a.status, (int32_t)KDA_ERR_TIMEOUT);
  sm100::tc_fence_after();
  if (ok) {
    for (int c = 0; c < N; c += 16) {
      float v[16];
      sm100::tmem_ld16(sm100::taddr(tbase, lane0, d_col + c), v);
      sm100::tmem_wait_ld();
      const int lane = lane0 + tid % 32;
#pragma unroll
      for (int i = 0; i < 16; ++i) a.D[lane * N + c + i] = v[i];
    }
  }
  sm100::tc_fence_before();
  __syncthreads();
  if (warp == 0) sm100::tmem_dealloc(tbase, 512);
}

}  // namespace

extern "C" kda_status kda_debug_umma(const uint16_t* A, const uint16_t* B, float* D, int M,
                                     int N, int K, int a_mode, int b_mode, int pack,
                                     int32_t* dev_status, kda_stream_t stream) {
  if (!A || !B || !D) return KDA_ERR_INVALID_ARG;
  if (M != 64 && M != 128) return KDA_ERR_UNSUPPORTED;
  if (K < 16 || K > 128 || K % 16) return KDA_ERR_UNSUPPORTED;
  if (N < 16 || N > 256 || N % 16) return KDA_ERR_UNSUPPORTED;
  if (a_mode < 0 || a_mode > 2 || b_mode < 0 || b_mode > 2 || pack < 0 || pack > 1)
    return KDA_ERR_INVALID_ARG;
  if (a_mode == 2 && M != 128) return KDA_ERR_UNSUPPORTED;
  if (b_mode == 2 && N != 64) return KDA_ERR_UNSUPPORTED;
  ProbeArgs p{A, B, D, dev_status, M, N, K, a_mode, b_mode, pack};
  const int smem = 32768 + 65536 + 65536;  // operands + slack
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaFuncSetAttribute(umma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return KDA_ERR_CUDA;
  umma_probe_kernel<<<1, kProbeThreads, smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
