// kda_tc_util.cuh -- device and host helpers shared by the tensor-core
// kernels: shared-memory operand layouts, bf16 packing, the decay map on the
// special-function unit, warp-level tf32 products for the triangular solve,
// and the TMA tensor maps over [rows, H, d] bf16 tensors.
#pragma once

#include <cudaTypedefs.h>
#include <string.h>

#include "kda_common.cuh"
#include "sm100.cuh"

namespace kda_tc {
// ---- operand layouts (core matrices of 8 x 16 B) ---------------------------
// MN-major: element (mn, k) with `lbo` the K-group stride, M/N groups 128 B apart
__device__ __forceinline__ uint32_t mn_off(int mn, int k, uint32_t lbo) {
  return (uint32_t)(mn >> 3) * 128u + (uint32_t)(k >> 3) * lbo + (uint32_t)(k & 7) * 16u +
         (uint32_t)(mn & 7) * 2u;
}
// K-major with K extent 64: K groups 128 B apart, M/N groups 1024 B apart
__device__ __forceinline__ uint32_t k64_off(int mn, int k) {
  return (uint32_t)(mn >> 3) * 1024u + (uint32_t)(k >> 3) * 128u + (uint32_t)(mn & 7) * 16u +
         (uint32_t)(k & 7) * 2u;
}
// 128B-swizzled TMA row: element (row, ch) of a [rows][64] bf16 box
__device__ __forceinline__ uint32_t sw128_off(int row, int ch) {
  return (uint32_t)row * 128u + (uint32_t)(((ch >> 3) ^ (row & 7)) << 4) + (uint32_t)(ch & 7) * 2u;
}
// unswizzled TMA row: element (row, ch) of a [rows][64] bf16 box (conflict-free
// as long as a warp reads along one row)
__device__ __forceinline__ uint32_t row_off(int row, int ch) {
  return (uint32_t)row * 128u + (uint32_t)ch * 2u;
}
__device__ __forceinline__ float ld_bf16(const unsigned char* base, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(base + off));
}

__device__ __forceinline__ void st16(unsigned char* p, uint32_t a, uint32_t b, uint32_t c,
                                     uint32_t d) {
  *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}
// pack 8 floats (v[0..7]) into a 16-byte chunk of bf16
__device__ __forceinline__ void st8_bf16(unsigned char* p, const float* v) {
  st16(p, sm100::pack_bf16x2(v[0], v[1]), sm100::pack_bf16x2(v[2], v[3]),
       sm100::pack_bf16x2(v[4], v[5]), sm100::pack_bf16x2(v[6], v[7]));
}

__device__ __forceinline__ float alpha_of(float x) {
  // exp(max(-softplus(x), -5)) = max(sigmoid(-x), e^-5) = max(1 / (1 + e^x), e^-5):
  // one ex2 and one rcp on the special-function unit (flush-to-zero is exact
  // here: e^x underflowing gives alpha = 1, overflowing gives the floor)
  float t, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(x * 1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + t));
  return fmaxf(r, 0.006737946999085467f);
}

// Warp-level m16n8k8 product, tf32 operands, fp32 accumulation, for the
// 16- and 32-row block merges of the triangular solve (far below the 64-row
// minimum of tcgen05.mma; T is rounded to bf16 afterwards, so tf32's 2^-11
// operand rounding stays below what the rest of the path keeps).
// Fragments (g = lane / 4, t = lane % 4):
//   a0 = A[g][t], a1 = A[g+8][t], a2 = A[g][t+4], a3 = A[g+8][t+4]
//   b0 = B[t][g], b1 = B[t+4][g];  d0 = D[g][2t], d1 = D[g][2t+1],
//   d2 = D[g+8][2t], d3 = D[g+8][2t+1]
__device__ __forceinline__ uint32_t tf32_of(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// D(16x8 tile) += A[a_row0.., a_col0 + k..] * B[b_row0 + k.., b_col0..] over
// k in [K0, K1) (multiples of 8, fixed at compile time so that every
// fragment load is issued ahead of the products); A, B fp32 row-major with
// leading dims.
template <int K0, int K1>
__device__ __forceinline__ void mma_tile(float (&d)[4], const float* A, int lda, int a_row0,
                                         int a_col0, const float* B, int ldb, int b_row0,
                                         int b_col0, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int k = K0; k < K1; k += 8) {
    uint32_t a[4], b[2];
    const float* Ar = A + (a_row0 + g) * lda + a_col0 + k + t;
    a[0] = tf32_of(Ar[0]);
    a[1] = tf32_of(Ar[8 * lda]);
    a[2] = tf32_of(Ar[4]);
    a[3] = tf32_of(Ar[8 * lda + 4]);
    const float* Bc = B + (b_row0 + k + t) * ldb + b_col0 + g;
    b[0] = tf32_of(Bc[0]);
    b[1] = tf32_of(Bc[4 * ldb]);
    mma_tf32(d, a, b);
  }
}
// store a 16x8 accumulator tile (scaled) at D[row0.., col0..]
__device__ __forceinline__ void store_tile(const float (&d)[4], float* D, int ldd, int row0,
                                           int col0, float sc, int lane) {
  const int g = lane >> 2, t = lane & 3;
  float* r0 = D + (row0 + g) * ldd + col0 + 2 * t;
  float* r1 = r0 + 8 * ldd;
  *reinterpret_cast<float2*>(r0) = make_float2(sc * d[0], sc * d[1]);
  *reinterpret_cast<float2*>(r1) = make_float2(sc * d[2], sc * d[3]);
}

// bf16 copy of a 16x8 accumulator tile into a K-major [r][i] operand with K
// extent 64 (one packed pair per row and lane), column c scaled by cs(c)
// times `sc`
template <class ColScale>
__device__ __forceinline__ void store_tile_bf16(const float (&d)[4], unsigned char* t, int row0,
                                                int col0, float sc, int lane, ColScale cs) {
  const int g = lane >> 2, c0 = col0 + 2 * (lane & 3);
  const float s0 = sc * cs(c0), s1 = sc * cs(c0 + 1);
  *reinterpret_cast<uint32_t*>(t + k64_off(row0 + g, c0)) =
      sm100::pack_bf16x2(s0 * d[0], s1 * d[1]);
  *reinterpret_cast<uint32_t*>(t + k64_off(row0 + g + 8, c0)) =
      sm100::pack_bf16x2(s0 * d[2], s1 * d[3]);
}

// column scales for unit_lower_inverse's bf16 output: none (T itself)
struct NoColScale {
  __device__ __forceinline__ float operator()(int) const { return 1.0f; }
};

// ---------------------------------------------------------------------------
// T = (I + A)^{-1} for a strictly lower triangular 64 x 64 fp32 matrix A
// (A = diag(beta) A_kk of one chunk), blocked by 16 x 16 tiles:
// (1) the four diagonal tiles, two warps each, one column per group of four
//     lanes, right-looking substitution in registers (critical path: 15
//     FMAs), lane q of a group owning rows q, q+4, q+8, q+12 and the pivot
//     arriving by shuffle;
// (2) T[2h+1, 2h] = -T[2h+1, 2h+1] (A[2h+1, 2h] T[2h, 2h]) for h = 0, 1, one
//     16 x 8 column tile per warp (warps 0-3), the inner product kept in
//     registers and turned into the outer product's operand by shuffles;
//     warps 4-7 meanwhile zero the tiles of T above the block diagonal;
// (3) T[H1, H0]  = -T[H1, H1] A[H1, H0] T[H0, H0] on the 32 x 32 halves.
// Each tile of T is written as bf16 by the step that makes it.
// Called by all 256 threads of the CTA (it synchronises them, but not after
// the last step).  A is read from `a` (row stride LD floats; blocks above
// the block diagonal are never read), the strictly lower part of T is left
// in `tf` (same stride), `y` ([32][36] fp32) is scratch, and T Diag(cs) (T
// with column i scaled by cs(i): unit diagonal times cs, zero above) is
// written as bf16 K-major [r][i] to `t_bf16`; the fp32 copy in `tf` is T
// itself.  LD is a multiple of 4 (rows are read as float4).
template <int LD, class ColScale = NoColScale>
__device__ __forceinline__ void unit_lower_inverse(const float* a, float* tf, float* y,
                                                   unsigned char* t_bf16, int tid,
                                                   ColScale cs = ColScale()) {
  static_assert(LD % 4 == 0, "row stride");
  const int warp = tid >> 5, lane = tid & 31;
  {
    const int blk = warp >> 1, c = (warp & 1) * 8 + (lane >> 2), q = lane & 3;
    const float* A = a + (16 * blk) * LD + 16 * blk;
    float a_reg[4][16];
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        const float4 v4 = *reinterpret_cast<const float4*>(A + (4 * k4 + q) * LD + 4 * i4);
        a_reg[k4][4 * i4] = v4.x; a_reg[k4][4 * i4 + 1] = v4.y;
        a_reg[k4][4 * i4 + 2] = v4.z; a_reg[k4][4 * i4 + 3] = v4.w;
      }
    }
    float x[4];
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) x[k4] = (4 * k4 + q == c) ? 1.0f : 0.0f;
    const int src0 = lane & ~3;
#pragma unroll
    for (int i = 0; i < 15; ++i) {
      const float xi = __shfl_sync(0xffffffffu, x[i >> 2], src0 | (i & 3));
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        if (4 * k4 + q > i) x[k4] = fmaf(-a_reg[k4][i], xi, x[k4]);
      }
    }
    const float csc = cs(16 * blk + c);
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const int r = 16 * blk + 4 * k4 + q;
      tf[r * LD + 16 * blk + c] = x[k4];
      *reinterpret_cast<__nv_bfloat16*>(t_bf16 + k64_off(r, 16 * blk + c)) =
          __float2bfloat16_rn(x[k4] * csc);
    }
  }
  __syncthreads();
  if (warp < 4) {
    // (2) warp w: h = w >> 1, 8-column tile w & 1
    const int hh = warp >> 1, nt = (warp & 1) * 8;
    const int a1 = 2 * hh + 1, a0 = 2 * hh;
    const int g = lane >> 2, t = lane & 3;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    // Y = A[2h+1, 2h] T[2h, 2h] (16 x 8 tile, accumulator layout)
    mma_tile<0, 16>(d, a, LD, 16 * a1, 16 * a0, tf, LD, 16 * a0, 16 * a0 + nt, lane);
    // operand fragments of Y for the second product: lane (g, t) takes
    // Y[t + 4u][g] (u = 0..3), held by lane 4 (t + 4u mod 8) + g / 2 as its
    // element 2 (u / 2) + g % 2
    const int s0 = 4 * t + (g >> 1), s1 = s0 + 16;
    float y0[4], y1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      y0[e] = __shfl_sync(0xffffffffu, d[e], s0);
      y1[e] = __shfl_sync(0xffffffffu, d[e], s1);
    }
    const bool odd = (g & 1) != 0;
    const uint32_t bk0[2] = {tf32_of(odd ? y0[1] : y0[0]), tf32_of(odd ? y1[1] : y1[0])};
    const uint32_t bk1[2] = {tf32_of(odd ? y0[3] : y0[2]), tf32_of(odd ? y1[3] : y1[2])};
    // T[2h+1, 2h] = -T[2h+1, 2h+1] Y
    float e2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const float* Ar = tf + (16 * a1 + g) * LD + 16 * a1 + 8 * ks + t;
      const uint32_t af[4] = {tf32_of(Ar[0]), tf32_of(Ar[8 * LD]), tf32_of(Ar[4]),
                              tf32_of(Ar[8 * LD + 4])};
      mma_tf32(e2, af, ks ? bk1 : bk0);
    }
    store_tile(e2, tf, LD, 16 * a1, 16 * a0 + nt, -1.0f, lane);
    store_tile_bf16(e2, t_bf16, 16 * a1, 16 * a0 + nt, -1.0f, lane, cs);
  } else {
    // zero the six 16 x 16 tiles above the block diagonal: 24 core matrices
    // of 128 bytes, written 16 bytes at a time
    for (int e = tid - 128; e < 24 * 8; e += 128) {
      const int cm = e >> 3, piece = e & 7, tix = cm >> 2, sub = cm & 3;
      const int R = tix < 3 ? 0 : (tix < 5 ? 1 : 2);
      const int I = tix < 3 ? tix + 1 : (tix < 5 ? tix - 1 : 3);
      *reinterpret_cast<uint4*>(t_bf16 + (2 * R + (sub >> 1)) * 1024 +
                                (2 * I + (sub & 1)) * 128 + piece * 16) =
          make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();
  // (3) level 2 on the 32 x 32 halves; warp w: rows 16 (w >> 2), columns 8 (w & 3)
  {
    const int mt = (warp >> 2) * 16, nt = (warp & 3) * 8;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    // Y = A[H1, H0] T[H0, H0] (T lower triangular: k from the tile's column;
    // the block above T's diagonal tiles is never written, so it is skipped)
    switch (nt >> 3) {
      case 0: mma_tile<0, 32>(d, a, LD, 32 + mt, 0, tf, LD, 0, nt, lane); break;
      case 1: mma_tile<8, 32>(d, a, LD, 32 + mt, 0, tf, LD, 0, nt, lane); break;
      case 2: mma_tile<16, 32>(d, a, LD, 32 + mt, 0, tf, LD, 0, nt, lane); break;
      default: mma_tile<24, 32>(d, a, LD, 32 + mt, 0, tf, LD, 0, nt, lane); break;
    }
    store_tile(d, y, 36, mt, nt, 1.0f, lane);
  }
  __syncthreads();
  {
    const int mt = (warp >> 2) * 16, nt = (warp & 3) * 8;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    // T[H1, H0] = -T[H1, H1] Y (T[H1, H1] lower triangular: k up to the row tile)
    if (mt == 0) mma_tile<0, 16>(d, tf, LD, 32, 32, y, 36, 0, nt, lane);
    else mma_tile<0, 32>(d, tf, LD, 48, 32, y, 36, 0, nt, lane);
    store_tile(d, tf, LD, 32 + mt, nt, -1.0f, lane);
    store_tile_bf16(d, t_bf16, 32 + mt, nt, -1.0f, lane, cs);
  }
}

// A CTA barrier (with the tensor-core ordering fences) that also makes every
// thread agree on whether any thread has recorded an error: a thread that
// runs ahead and fails a later wait cannot make the others leave the loop
// at different points.
__device__ __forceinline__ bool sync_aborted(const int* s_abort) {
  sm100::tc_fence_before();
  const int any = __syncthreads_or(*reinterpret_cast<const volatile int*>(s_abort));
  sm100::tc_fence_after();
  return any != 0;
}

// ---------------------------------------------------------------------------
// host: TMA tensor maps
inline PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 3-D map over a [rows, H, d] bf16 tensor: box = box_ch channels x 1 head x 64
// rows, rows 128B-swizzled in shared memory unless `swizzle` is false (a box
// of 8 channels, unswizzled, lands as 64 rows of 16 bytes: one column of
// core matrices of an MN-major operand whose K index is the row)
inline bool make_map(CUtensorMap* m, const void* base, int64_t rows, int H, int d,
                     bool swizzle = true, int box_ch = 64) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_ch, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace kda_tc
