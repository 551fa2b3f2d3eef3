// elementwise.cu -- HBM-bound kernels of the NVFP4 MoE path: quantiser
// (with the warp-shuffle tensor amax), weight-scale packing, SwiGLU +
// requantisation, and the weighted combine; their MXFP4 counterparts; and the
// FP8 (E4M3, per-tensor scale) activation quantisers of the W4A8 mode.
//
// All of them are one-pass streaming kernels: coalesced 16-byte loads and
// stores, grids sized in multiples of the SM count, no shared-memory staging
// (nothing is reused).
#include "common.cuh"
#include "kernels.h"

namespace nvfp4moe {

// ---------------------------------------------------------------------------
// tensor amax (dynamic per-tensor scale)
// ---------------------------------------------------------------------------

// Eight consecutive inputs widened to fp32 (16- or 32-byte aligned load).
template <typename T>
__device__ __forceinline__ void load8(const T* p, float* v);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float* v) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, float* v) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// amax over [rows, cols] (cols % 8 == 0) -> atomicMax on the bit pattern
// (|x| >= 0, so unsigned order equals float order).
template <typename T>
__global__ void __launch_bounds__(256) amax_kernel(const T* __restrict__ x, int64_t rows, int64_t cols,
                                                   int64_t ld, uint32_t* __restrict__ amax_bits) {
  pdl_wait();
  pdl_trigger();
  const int64_t vec_per_row = cols / 8;
  const int64_t nvec = rows * vec_per_row;
  float m = 0.0f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / vec_per_row, c = (i % vec_per_row) * 8;
    float v[8];
    load8<T>(x + r * ld + c, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ float wmax[8];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) b = fmaxf(b, wmax[w]);
    atomicMax(amax_bits, __float_as_uint(b));
  }
}

// One thread per 16-element block.  dynamic: S = amax / 2688 from the amax
// word; static: S read from *S.
template <typename T>
__global__ void __launch_bounds__(256) quantize_kernel(const T* __restrict__ x, int64_t rows, int64_t cols,
                                                       int64_t ld, float* __restrict__ S, int dynamic,
                                                       const uint32_t* __restrict__ amax_bits,
                                                       uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  float s;
  if (dynamic) {
    s = __fdiv_rn(__uint_as_float(*amax_bits), 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *S = s;
  } else {
    s = *S;
  }
  const int64_t nb_row = cols / 16;
  const int64_t nblk = rows * nb_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nblk; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nb_row, b = i % nb_row;
    float v[16];
    load8<T>(x + r * ld + b * 16, v);
    load8<T>(x + r * ld + b * 16 + 8, v + 8);
    uint32_t w0, w1;
    const uint32_t sc = quantize_block16(v, s, w0, w1);
    *reinterpret_cast<uint2*>(codes + r * (cols / 2) + b * 8) = make_uint2(w0, w1);
    scales[r * nb_row + b] = (uint8_t)sc;
  }
}

// Quantise x [T, H] (bf16) with the dynamic scale S = amax / 2688 and write
// every token's NVFP4 row straight to its k permuted rows inv[t*k + j]: the
// quantiser and the row gather in one pass (each block quantised once).
__global__ void __launch_bounds__(256) quantize_scatter_kernel(const __nv_bfloat16* __restrict__ x, int T, int64_t H,
                                                               int k, const int32_t* __restrict__ inv,
                                                               const uint32_t* __restrict__ amax_bits,
                                                               float* __restrict__ S, uint8_t* __restrict__ codes,
                                                               uint8_t* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  const float s = __fdiv_rn(__uint_as_float(*amax_bits), 2688.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *S = s;
  const int64_t nb_row = H / 16;
  const int64_t nblk = (int64_t)T * nb_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nblk; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / nb_row, b = i % nb_row;
    float v[16];
    load8<__nv_bfloat16>(x + t * H + b * 16, v);
    load8<__nv_bfloat16>(x + t * H + b * 16 + 8, v + 8);
    uint32_t w0, w1;
    const uint8_t sc = (uint8_t)quantize_block16(v, s, w0, w1);
    for (int j = 0; j < k; ++j) {
      const int64_t r = __ldg(inv + t * k + j);
      *reinterpret_cast<uint2*>(codes + r * (H / 2) + b * 8) = make_uint2(w0, w1);
      scales[r * nb_row + b] = sc;
    }
  }
}

// ---------------------------------------------------------------------------
// FP8 (E4M3) activations with a per-tensor decode scale (the W4A8 mode)
// ---------------------------------------------------------------------------

// FP8 activation code of x with decode scale s: the sign bit of x / s, then
// E4M3(RNE, satfinite) of |x / s|; s == 0 gives code 0.
__device__ __forceinline__ uint32_t fp8_code(float x, float s) {
  if (s == 0.0f) return 0;
  const float q = __fdiv_rn(x, s);
  return e4m3_from_f32(fabsf(q)) | ((__float_as_uint(q) >> 31) << 7);
}

// Two FP8 codes (low byte: the lower element) -> their values as f16x2 (exact:
// every E4M3 value is an f16).
__device__ __forceinline__ uint32_t f16x2_of_e4m3x2(uint32_t two) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)two));
  return d;
}
// Eight FP8 codes (two words) -> their eight f16 values (four words).
__device__ __forceinline__ uint4 f16x8_of_e4m3x8(uint2 c) {
  return make_uint4(f16x2_of_e4m3x2(c.x & 0xFFFFu), f16x2_of_e4m3x2(c.x >> 16), f16x2_of_e4m3x2(c.y & 0xFFFFu),
                    f16x2_of_e4m3x2(c.y >> 16));
}

// Eight inputs -> eight FP8 codes (two little-endian words), decode scale s.
__device__ __forceinline__ uint2 fp8_codes8(const float (&v)[8], float s) {
  uint32_t w[2];
#pragma unroll
  for (int q = 0; q < 2; ++q)
    w[q] = fp8_code(v[4 * q], s) | (fp8_code(v[4 * q + 1], s) << 8) | (fp8_code(v[4 * q + 2], s) << 16) |
           (fp8_code(v[4 * q + 3], s) << 24);
  return make_uint2(w[0], w[1]);
}

// One thread per 8 elements.  dynamic: S = amax / 448 from the amax word;
// static: S read from *S.
template <typename T>
__global__ void __launch_bounds__(256) fp8_quantize_kernel(const T* __restrict__ x, int64_t rows, int64_t cols,
                                                           int64_t ld, float* __restrict__ S, int dynamic,
                                                           const uint32_t* __restrict__ amax_bits,
                                                           uint8_t* __restrict__ codes) {
  pdl_wait();
  pdl_trigger();
  float s;
  if (dynamic) {
    s = __fdiv_rn(__uint_as_float(*amax_bits), 448.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *S = s;
  } else {
    s = *S;
  }
  const int64_t nv_row = cols / 8;
  const int64_t nv = rows * nv_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nv; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nv_row, c = (i % nv_row) * 8;
    float v[8];
    load8<T>(x + r * ld + c, v);
    *reinterpret_cast<uint2*>(codes + r * cols + c) = fp8_codes8(v, s);
  }
}

// Quantise x [T, H] (bf16) to FP8 with the dynamic scale S = amax / 448 and
// write every token's row straight to its k permuted rows inv[t*k + j].
__global__ void __launch_bounds__(256) fp8_quantize_scatter_kernel(const __nv_bfloat16* __restrict__ x, int T,
                                                                   int64_t H, int k, const int32_t* __restrict__ inv,
                                                                   const uint32_t* __restrict__ amax_bits,
                                                                   float* __restrict__ S,
                                                                   uint8_t* __restrict__ codes,
                                                                   __half* __restrict__ f16_out,
                                                                   float* __restrict__ rs) {
  pdl_wait();
  pdl_trigger();
  const float s = __fdiv_rn(__uint_as_float(*amax_bits), 448.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *S = s;
  const int64_t nv_row = H / 8;
  const int64_t nv = (int64_t)T * nv_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nv; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / nv_row, c = (i % nv_row) * 8;
    float v[8];
    load8<__nv_bfloat16>(x + t * H + c, v);
    const uint2 w = fp8_codes8(v, s);
    if (f16_out == nullptr) {
      for (int j = 0; j < k; ++j) *reinterpret_cast<uint2*>(codes + (int64_t)__ldg(inv + t * k + j) * H + c) = w;
    } else {
      // the F16 carrier: each code's value (exact), the scale per row
      const uint4 f = f16x8_of_e4m3x8(w);
      for (int j = 0; j < k; ++j) {
        const int64_t r = __ldg(inv + t * k + j);
        *reinterpret_cast<uint4*>(f16_out + r * H + c) = f;
        if (c == 0) rs[r] = s;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// weight-scale packing: linear [E, N, K/16] -> 512-byte atoms
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) pack_scales_kernel(const uint8_t* __restrict__ in, int64_t E, int64_t N,
                                                          int64_t K, uint8_t* __restrict__ out) {
  const int64_t kb_n = K / 64;                  // 4-scale words per row
  const int64_t total = E * N * kb_n;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / kb_n, kb = i % kb_n;   // row = e*N + n
    const int64_t e = row / N, n = row % N;
    const uint32_t word = *reinterpret_cast<const uint32_t*>(in + row * (K / 16) + kb * 4);
    const int64_t nt = n / 128, r = n % 128;
    const int64_t atom = (e * (N / 128) + nt) * kb_n + kb;
    *reinterpret_cast<uint32_t*>(out + atom * 512 + (r % 32) * 16 + (r / 32) * 4) = word;
  }
}

// ---------------------------------------------------------------------------
// SwiGLU + requantisation (one thread per 16-element block of h)
// ---------------------------------------------------------------------------

__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

__global__ void __launch_bounds__(256) swiglu_requant_kernel(const float* __restrict__ G, int64_t R, int64_t I,
                                                             int mode, const float* __restrict__ S_h,
                                                             uint8_t* __restrict__ h_codes,
                                                             uint8_t* __restrict__ h_scales,
                                                             __nv_bfloat16* __restrict__ h_bf16,
                                                             __half* __restrict__ h_f16, float* __restrict__ h_rs) {
  pdl_wait();
  pdl_trigger();
  const int64_t nb_row = I / 16;
  const int64_t nblk = R * nb_row;
  const float s = (mode == MOE_W4A4 || mode == MOE_W4A8) ? *S_h : 0.0f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nblk; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nb_row, b = i % nb_row;
    const float4* gp = reinterpret_cast<const float4*>(G + r * 2 * I + b * 16);
    const float4* up = reinterpret_cast<const float4*>(G + r * 2 * I + I + b * 16);
    float h[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 g = __ldg(gp + q), u = __ldg(up + q);
      h[4 * q + 0] = silu_mul(g.x, u.x);
      h[4 * q + 1] = silu_mul(g.y, u.y);
      h[4 * q + 2] = silu_mul(g.z, u.z);
      h[4 * q + 3] = silu_mul(g.w, u.w);
    }
    if (mode == MOE_W4A4) {
      uint32_t w0, w1;
      const uint32_t sc = quantize_block16(h, s, w0, w1);
      *reinterpret_cast<uint2*>(h_codes + r * (I / 2) + b * 8) = make_uint2(w0, w1);
      h_scales[r * nb_row + b] = (uint8_t)sc;
    } else if (mode == MOE_W4A8) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = fp8_code(h[4 * q], s) | (fp8_code(h[4 * q + 1], s) << 8) | (fp8_code(h[4 * q + 2], s) << 16) |
               (fp8_code(h[4 * q + 3], s) << 24);
      if (h_f16 == nullptr) {
        *reinterpret_cast<uint4*>(h_codes + r * I + b * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      } else {
        // the F16 carrier of the FP8 codes: their values (exact), the scale per row
        uint4* dst = reinterpret_cast<uint4*>(h_f16 + r * I + b * 16);
        dst[0] = f16x8_of_e4m3x8(make_uint2(w[0], w[1]));
        dst[1] = f16x8_of_e4m3x8(make_uint2(w[2], w[3]));
        if (b == 0) h_rs[r] = s;
      }
    } else {
      uint32_t w[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(h[2 * q], h[2 * q + 1]);
        w[q] = *reinterpret_cast<const uint32_t*>(&p);
      }
      uint4* dst = reinterpret_cast<uint4*>(h_bf16 + r * I + b * 16);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

// ---------------------------------------------------------------------------
// combine: out[t, n] = sum_j w[t, j] * Y[inv[t*k + j], n]  (gather, fp32)
// ---------------------------------------------------------------------------

// inv comes from the caller: a row outside [0, T*k) contributes nothing and
// is reported as NVFP4_E_BAD_ROUTING (never read).
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ Y, const int32_t* __restrict__ inv,
                                                      const float* __restrict__ w, int T, int k, int64_t H, int cs,
                                                      int out_dtype, void* __restrict__ out, int32_t* dev_status) {
  // block b: token b / cs, the (b % cs)-th of cs column ranges of its row.
  // The token's k row indices and weights are read once per block into
  // shared memory (a row outside [0, T*k) is marked -1); each thread then
  // keeps the k row loads of two float4 columns in flight.
  __shared__ int64_t s_r[32];
  __shared__ float s_w[32];
  pdl_wait();
  pdl_trigger();
  const int64_t q_per_row = H / 4;
  const int64_t chunk = (q_per_row + cs - 1) / cs;
  const uint32_t R = (uint32_t)T * (uint32_t)k;
  for (int64_t b = blockIdx.x; b < (int64_t)T * cs; b += gridDim.x) {
    const int64_t t = b / cs;
    const int64_t q0 = (b % cs) * chunk, q1 = min(q_per_row, q0 + chunk);
    __syncthreads();  // the previous token's s_r / s_w have been read
    if (threadIdx.x < k) {
      const int32_t rr = __ldg(inv + t * k + threadIdx.x);
      const bool ok = (uint32_t)rr < R;
      if (!ok) report_status(dev_status, NVFP4_E_BAD_ROUTING);
      s_r[threadIdx.x] = ok ? (int64_t)rr * H : -1;
      s_w[threadIdx.x] = __ldg(w + t * k + threadIdx.x);
    }
    __syncthreads();
    for (int64_t q = q0 + threadIdx.x; q < q1; q += 2 * (int64_t)blockDim.x) {
      const int64_t c0 = q * 4, c1 = (q + blockDim.x) * 4;
      const bool two = q + blockDim.x < q1;
      float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
      // rows in chunks of 8 (loads issued together; the sum runs in j order)
      for (int j0 = 0; j0 < k; j0 += 8) {
        float4 y0[8], y1[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int64_t r = (j0 + j < k) ? s_r[j0 + j] : -1;
          if (r >= 0) {
            y0[j] = __ldg(reinterpret_cast<const float4*>(Y + r + c0));
            if (two) y1[j] = __ldg(reinterpret_cast<const float4*>(Y + r + c1));
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int64_t r = (j0 + j < k) ? s_r[j0 + j] : -1;
          if (r >= 0) {
            const float wj = s_w[j0 + j];
            a0.x = __fadd_rn(a0.x, __fmul_rn(wj, y0[j].x));
            a0.y = __fadd_rn(a0.y, __fmul_rn(wj, y0[j].y));
            a0.z = __fadd_rn(a0.z, __fmul_rn(wj, y0[j].z));
            a0.w = __fadd_rn(a0.w, __fmul_rn(wj, y0[j].w));
            if (two) {
              a1.x = __fadd_rn(a1.x, __fmul_rn(wj, y1[j].x));
              a1.y = __fadd_rn(a1.y, __fmul_rn(wj, y1[j].y));
              a1.z = __fadd_rn(a1.z, __fmul_rn(wj, y1[j].z));
              a1.w = __fadd_rn(a1.w, __fmul_rn(wj, y1[j].w));
            }
          }
        }
      }
      for (int u = 0; u < (two ? 2 : 1); ++u) {
        const float4 acc = u ? a1 : a0;
        const int64_t c = u ? c1 : c0;
        if (out_dtype == NVFP4_DT_F32) {
          *reinterpret_cast<float4*>(static_cast<float*>(out) + t * H + c) = acc;
        } else {
          const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
          const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
          uint2 v;
          v.x = *reinterpret_cast<const uint32_t*>(&lo);
          v.y = *reinterpret_cast<const uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + t * H + c) = v;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// MXFP4: quantiser, quantise-scatter, weight-scale packing, SwiGLU + requant
// (one thread per 32-element block; scale rows padded to mx_scale_pitch)
// ---------------------------------------------------------------------------

template <typename T>
__global__ void __launch_bounds__(256) mx_quantize_kernel(const T* __restrict__ x, int64_t rows, int64_t cols,
                                                          int64_t ld, uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  const int64_t nb = cols / 32, pitch = mx_scale_pitch(cols);
  const int64_t total = rows * pitch;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / pitch, b = i % pitch;
    if (b >= nb) {
      scales[i] = 0;  // row padding
      continue;
    }
    float v[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) load8<T>(x + r * ld + b * 32 + 8 * q, v + 8 * q);
    uint4 c;
    const uint32_t sc = mx_quantize_block32(v, c);
    *reinterpret_cast<uint4*>(codes + r * (cols / 2) + b * 16) = c;
    scales[i] = (uint8_t)sc;
  }
}

__global__ void __launch_bounds__(256) mx_quantize_scatter_kernel(const __nv_bfloat16* __restrict__ x, int T,
                                                                  int64_t H, int k, const int32_t* __restrict__ inv,
                                                                  uint8_t* __restrict__ codes,
                                                                  uint8_t* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  const int64_t nb = H / 32, pitch = mx_scale_pitch(H);
  const int64_t total = (int64_t)T * pitch;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / pitch, b = i % pitch;
    if (b >= nb) {
      for (int j = 0; j < k; ++j) scales[(int64_t)__ldg(inv + t * k + j) * pitch + b] = 0;
      continue;
    }
    float v[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) load8<__nv_bfloat16>(x + t * H + b * 32 + 8 * q, v + 8 * q);
    uint4 c;
    const uint8_t sc = (uint8_t)mx_quantize_block32(v, c);
    for (int j = 0; j < k; ++j) {
      const int64_t r = __ldg(inv + t * k + j);
      *reinterpret_cast<uint4*>(codes + r * (H / 2) + b * 16) = c;
      scales[r * pitch + b] = sc;
    }
  }
}

__global__ void __launch_bounds__(256) mx_pack_scales_kernel(const uint8_t* __restrict__ in, int64_t E, int64_t N,
                                                             int64_t K, uint8_t* __restrict__ out) {
  const int64_t kb_n = K / 64;  // scale pairs per row
  const int64_t total = E * N * kb_n;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / kb_n, kb = i % kb_n;  // row = e*N + n
    const int64_t e = row / N, n = row % N;
    const uint16_t pair = *reinterpret_cast<const uint16_t*>(in + row * (K / 32) + kb * 2);
    const int64_t nt = n / 128, r = n % 128;
    const int64_t blk = (e * (N / 128) + nt) * kb_n + kb;
    *reinterpret_cast<uint16_t*>(out + blk * 256 + (r % 32) * 8 + (r / 32) * 2) = pair;
  }
}

__global__ void __launch_bounds__(256) swiglu_requant_mx_kernel(const float* __restrict__ G, int64_t R, int64_t I,
                                                                uint8_t* __restrict__ h_codes,
                                                                uint8_t* __restrict__ h_scales) {
  pdl_wait();
  pdl_trigger();
  const int64_t nb = I / 32, pitch = mx_scale_pitch(I);
  const int64_t total = R * pitch;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / pitch, b = i % pitch;
    if (b >= nb) {
      h_scales[i] = 0;
      continue;
    }
    const float4* gp = reinterpret_cast<const float4*>(G + r * 2 * I + b * 32);
    const float4* up = reinterpret_cast<const float4*>(G + r * 2 * I + I + b * 32);
    float h[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 g = __ldg(gp + q), u = __ldg(up + q);
      h[4 * q + 0] = silu_mul(g.x, u.x);
      h[4 * q + 1] = silu_mul(g.y, u.y);
      h[4 * q + 2] = silu_mul(g.z, u.z);
      h[4 * q + 3] = silu_mul(g.w, u.w);
    }
    uint4 c;
    const uint32_t sc = mx_quantize_block32(h, c);
    *reinterpret_cast<uint4*>(h_codes + r * (I / 2) + b * 16) = c;
    h_scales[i] = (uint8_t)sc;
  }
}

// ---------------------------------------------------------------------------
// host -> device staging of a layer's inputs (page-locked host memory read by
// SM loads over the host link): range 0 in 16-byte units, range 1 in 4-byte
// units.  Each thread keeps kStageILP loads in flight before it stores, so
// the copy costs a few link round trips rather than one per element.
// ---------------------------------------------------------------------------

constexpr int kStageILP = 4;

__global__ void __launch_bounds__(256) stage_in_kernel(const uint4* s0, uint4* __restrict__ d0, int64_t n0,
                                                       const uint32_t* s1, uint32_t* __restrict__ d1, int64_t n1) {
  pdl_wait();
  pdl_trigger();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  for (int64_t i = t; i < n0; i += kStageILP * stride) {
    uint4 v[kStageILP];
#pragma unroll
    for (int u = 0; u < kStageILP; ++u)
      if (i + u * stride < n0) v[u] = s0[i + u * stride];
#pragma unroll
    for (int u = 0; u < kStageILP; ++u)
      if (i + u * stride < n0) d0[i + u * stride] = v[u];
  }
  for (int64_t i = t; i < n1; i += kStageILP * stride) {
    uint32_t v[kStageILP];
#pragma unroll
    for (int u = 0; u < kStageILP; ++u)
      if (i + u * stride < n1) v[u] = s1[i + u * stride];
#pragma unroll
    for (int u = 0; u < kStageILP; ++u)
      if (i + u * stride < n1) d1[i + u * stride] = v[u];
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

static int grid_for(int64_t work_items, int threads) {
  const int64_t blocks = (work_items + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms() * 8;   // a few waves of resident CTAs
  return (int)(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

cudaError_t launch_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld, float* S,
                            int dynamic, uint32_t* amax_ws, uint8_t* codes, uint8_t* scales, cudaStream_t st) {
  if (rows == 0) {
    if (dynamic) return cudaMemsetAsync(S, 0, sizeof(float), st);
    return cudaSuccess;
  }
  if (dynamic) {
    cudaError_t e = cudaMemsetAsync(amax_ws, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    const int g = grid_for(rows * cols / 8, 256);
    if (x_dtype == NVFP4_DT_BF16)
      e = launch_pdl(amax_kernel<__nv_bfloat16>, g, 256, 0, st, static_cast<const __nv_bfloat16*>(x), rows, cols, ld,
                     amax_ws);
    else
      e = launch_pdl(amax_kernel<float>, g, 256, 0, st, static_cast<const float*>(x), rows, cols, ld, amax_ws);
    if (e != cudaSuccess) return e;
  }
  const int g = grid_for(rows * cols / 16, 256);
  if (x_dtype == NVFP4_DT_BF16)
    return launch_pdl(quantize_kernel<__nv_bfloat16>, g, 256, 0, st, static_cast<const __nv_bfloat16*>(x), rows,
                      cols, ld, S, dynamic, static_cast<const uint32_t*>(amax_ws), codes, scales);
  return launch_pdl(quantize_kernel<float>, g, 256, 0, st, static_cast<const float*>(x), rows, cols, ld, S, dynamic,
                    static_cast<const uint32_t*>(amax_ws), codes, scales);
}

cudaError_t launch_quantize_scatter(const void* x_bf16, int T, int H, int k, const int32_t* inv,
                                    const uint32_t* amax_bits, float* S, uint8_t* codes, uint8_t* scales,
                                    cudaStream_t st) {
  const int64_t nblk = (int64_t)T * (H / 16);
  if (nblk == 0) return cudaSuccess;
  return launch_pdl(quantize_scatter_kernel, grid_for(nblk, 256), 256, 0, st, static_cast<const __nv_bfloat16*>(x_bf16),
                    T, (int64_t)H, k, inv, amax_bits, S, codes, scales);
}

cudaError_t launch_fp8_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld, float* S,
                                int dynamic, uint32_t* amax_ws, uint8_t* codes, cudaStream_t st) {
  if (rows == 0) {
    if (dynamic) return cudaMemsetAsync(S, 0, sizeof(float), st);
    return cudaSuccess;
  }
  if (dynamic) {
    cudaError_t e = cudaMemsetAsync(amax_ws, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    const int g = grid_for(rows * cols / 8, 256);
    if (x_dtype == NVFP4_DT_BF16)
      e = launch_pdl(amax_kernel<__nv_bfloat16>, g, 256, 0, st, static_cast<const __nv_bfloat16*>(x), rows, cols, ld,
                     amax_ws);
    else
      e = launch_pdl(amax_kernel<float>, g, 256, 0, st, static_cast<const float*>(x), rows, cols, ld, amax_ws);
    if (e != cudaSuccess) return e;
  }
  const int g = grid_for(rows * cols / 8, 256);
  if (x_dtype == NVFP4_DT_BF16)
    return launch_pdl(fp8_quantize_kernel<__nv_bfloat16>, g, 256, 0, st, static_cast<const __nv_bfloat16*>(x), rows,
                      cols, ld, S, dynamic, static_cast<const uint32_t*>(amax_ws), codes);
  return launch_pdl(fp8_quantize_kernel<float>, g, 256, 0, st, static_cast<const float*>(x), rows, cols, ld, S,
                    dynamic, static_cast<const uint32_t*>(amax_ws), codes);
}

cudaError_t launch_fp8_quantize_scatter(const void* x_bf16, int T, int H, int k, const int32_t* inv,
                                        const uint32_t* amax_bits, float* S, uint8_t* codes, cudaStream_t st,
                                        void* f16_out, float* rs) {
  const int64_t nv = (int64_t)T * (H / 8);
  if (nv == 0) return cudaSuccess;
  return launch_pdl(fp8_quantize_scatter_kernel, grid_for(nv, 256), 256, 0, st,
                    static_cast<const __nv_bfloat16*>(x_bf16), T, (int64_t)H, k, inv, amax_bits, S, codes,
                    static_cast<__half*>(f16_out), rs);
}

cudaError_t launch_pack_scales(const uint8_t* in, int E, int N, int K, uint8_t* out, cudaStream_t st) {
  const int64_t total = (int64_t)E * N * (K / 64);
  if (total == 0) return cudaSuccess;
  pack_scales_kernel<<<grid_for(total, 256), 256, 0, st>>>(in, E, N, K, out);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_requant(const float* G, int R, int I, int mode, const float* S_h, uint8_t* h_codes,
                                  uint8_t* h_scales, void* h_bf16, cudaStream_t st) {
  const int64_t nblk = (int64_t)R * (I / 16);
  if (nblk == 0) return cudaSuccess;
  return launch_pdl(swiglu_requant_kernel, grid_for(nblk, 256), 256, 0, st, G, (int64_t)R, (int64_t)I, mode, S_h,
                    h_codes, h_scales, static_cast<__nv_bfloat16*>(h_bf16), static_cast<__half*>(nullptr),
                    static_cast<float*>(nullptr));
}

cudaError_t launch_swiglu_fp8_f16(const float* G, int R, int I, const float* S_h, void* h_f16, float* h_rs,
                                  cudaStream_t st) {
  const int64_t nblk = (int64_t)R * (I / 16);
  if (nblk == 0) return cudaSuccess;
  return launch_pdl(swiglu_requant_kernel, grid_for(nblk, 256), 256, 0, st, G, (int64_t)R, (int64_t)I,
                    (int)MOE_W4A8, S_h, static_cast<uint8_t*>(nullptr), static_cast<uint8_t*>(nullptr),
                    static_cast<__nv_bfloat16*>(nullptr), static_cast<__half*>(h_f16), h_rs);
}

// ---------------------------------------------------------------------------
// F16 carrier of BF16 rows (the W4A16 product on F16 tensor-core operands).
// A bf16 value has 8 significant bits, an f16 11, but f16 spans only
// [2^-24, 65504].  Row r is carried as f16(x * 2^e_r) with the power of two
// chosen so that the row's max |x| lands in [2^14, 2^15): every element of
// the row within a factor 2^28 of that max stays an f16 normal and is exact;
// smaller ones round to the f16 subnormal grid, an absolute error of at most
// 2^-39 times the row's max.  rs[r] = 2^-e_r undoes the scaling (exactly:
// a power of two) in the GEMM's epilogue.
// ---------------------------------------------------------------------------

// e_r for a row whose largest magnitude is amax (0: an all-zero row), kept
// within [-113, 126] so that 2^e and 2^-e are fp32 normals.
__device__ __forceinline__ int f16_row_exponent(float amax) {
  if (!(amax > 0.0f)) return 0;
  const int e = 14 - ilogbf(amax);
  return e > 126 ? 126 : e;
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// The largest value of v over the block (256 threads), in every thread.
__device__ __forceinline__ float block_max256(float v) {
  __shared__ float red[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  __syncthreads();  // red[] of a previous call has been read
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  v = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) v = fmaxf(v, red[i]);
  return v;
}

// One 256-thread block per output row: a_f16[r] = x[src] * 2^e_r, rs[r] =
// 2^-e_r, with src = perm[r] (or r).  Two passes over the row (max, then
// convert); the second reads it from L1/L2.  (A warp per row left most SMs
// idle at decode sizes: 128 rows.)
__global__ void __launch_bounds__(256) gather_f16_kernel(const __nv_bfloat16* __restrict__ x, int64_t H,
                                                         const int32_t* __restrict__ perm, int R,
                                                         __half* __restrict__ a, float* __restrict__ rs) {
  pdl_wait();
  pdl_trigger();
  for (int64_t r = blockIdx.x; r < R; r += gridDim.x) {
    const int64_t t = perm != nullptr ? (int64_t)__ldg(perm + r) : r;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
    float m = 0.0f;
    for (int64_t i = threadIdx.x; i < H / 8; i += blockDim.x) {
      const uint4 u = __ldg(src + i);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[q] << 16)), fabsf(__uint_as_float(w[q] & 0xFFFF0000u))));
    }
    m = block_max256(m);
    const int e = f16_row_exponent(m);
    const float sc = pow2f(e);
    uint4* dst = reinterpret_cast<uint4*>(a + r * H);
    for (int64_t i = threadIdx.x; i < H / 8; i += blockDim.x) {
      const uint4 u = __ldg(src + i);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t o4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __half2 h2 = __floats2half2_rn(__fmul_rn(__uint_as_float(w[q] << 16), sc),
                                             __fmul_rn(__uint_as_float(w[q] & 0xFFFF0000u), sc));
        o4[q] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      dst[i] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
    if (threadIdx.x == 0) rs[r] = pow2f(-e);
  }
}

// One 256-thread block per row r of G [R, 2I] (gate | up): h = bf16(silu(g)
// * u) -- the W4A16 activation of the down GEMM -- carried as f16(h * 2^e_r),
// rs[r] = 2^-e_r.  The bf16 values are written first (as 16-bit words into
// the f16 buffer) with the row's max taken on the way, then converted in
// place by the thread that wrote them.
__global__ void __launch_bounds__(256) swiglu_f16_kernel(const float* __restrict__ G, int64_t R, int64_t I,
                                                         __half* __restrict__ h, float* __restrict__ rs) {
  pdl_wait();
  pdl_trigger();
  for (int64_t r = blockIdx.x; r < R; r += gridDim.x) {
    const float4* gp = reinterpret_cast<const float4*>(G + r * 2 * I);
    const float4* up = reinterpret_cast<const float4*>(G + r * 2 * I + I);
    uint2* hrow = reinterpret_cast<uint2*>(h + r * I);
    float m = 0.0f;
    for (int64_t i = threadIdx.x; i < I / 4; i += blockDim.x) {
      const float4 g = __ldg(gp + i), u = __ldg(up + i);
      const __nv_bfloat162 b0 = __floats2bfloat162_rn(silu_mul(g.x, u.x), silu_mul(g.y, u.y));
      const __nv_bfloat162 b1 = __floats2bfloat162_rn(silu_mul(g.z, u.z), silu_mul(g.w, u.w));
      const uint32_t w0 = *reinterpret_cast<const uint32_t*>(&b0), w1 = *reinterpret_cast<const uint32_t*>(&b1);
      m = fmaxf(m, fmaxf(fmaxf(fabsf(__uint_as_float(w0 << 16)), fabsf(__uint_as_float(w0 & 0xFFFF0000u))),
                         fmaxf(fabsf(__uint_as_float(w1 << 16)), fabsf(__uint_as_float(w1 & 0xFFFF0000u)))));
      hrow[i] = make_uint2(w0, w1);
    }
    m = block_max256(m);  // then each thread converts the words it wrote
    const int e = f16_row_exponent(m);
    const float sc = pow2f(e);
    for (int64_t i = threadIdx.x; i < I / 4; i += blockDim.x) {
      const uint2 v = hrow[i];
      const __half2 h0 = __floats2half2_rn(__fmul_rn(__uint_as_float(v.x << 16), sc),
                                           __fmul_rn(__uint_as_float(v.x & 0xFFFF0000u), sc));
      const __half2 h1 = __floats2half2_rn(__fmul_rn(__uint_as_float(v.y << 16), sc),
                                           __fmul_rn(__uint_as_float(v.y & 0xFFFF0000u), sc));
      hrow[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
    }
    if (threadIdx.x == 0) rs[r] = pow2f(-e);
  }
}

cudaError_t launch_gather_f16(const void* x_bf16, int64_t H, const int32_t* perm, int R, void* a_f16, float* rs,
                              cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  return launch_pdl(gather_f16_kernel, R < 8 * num_sms() ? R : 8 * num_sms(), 256, 0, st,
                    static_cast<const __nv_bfloat16*>(x_bf16), H, perm, R, static_cast<__half*>(a_f16), rs);
}

cudaError_t launch_swiglu_f16(const float* G, int R, int I, void* h_f16, float* rs, cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  return launch_pdl(swiglu_f16_kernel, R < 8 * num_sms() ? R : 8 * num_sms(), 256, 0, st, G, (int64_t)R, (int64_t)I,
                    static_cast<__half*>(h_f16), rs);
}

// Zero fill of a GEMM's fp32 output before its K parts add into it.  An
// ordinary launch (it starts once the stream's previous work is complete)
// that lets the GEMM -- a programmatic dependent -- launch as soon as every
// block has started, so the GEMM's prologue overlaps the fill where a memset
// node would serialise the two launches.  (Launched as a programmatic
// dependent itself, its blocks would sit resident beside the previous kernel
// until that one completed; on GB300 that measured slower than a memset at
// 4-8 MB.)
__global__ void __launch_bounds__(256) zero_f32_kernel(float* __restrict__ p, size_t n) {
  pdl_trigger();
  const size_t n4 = n / 4, stride = (size_t)gridDim.x * blockDim.x;
  float4* p4 = reinterpret_cast<float4*>(p);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride)
    p4[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (size_t i = n4 * 4 + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = 0.0f;
}

cudaError_t launch_zero_f32(float* p, size_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return cudaMemsetAsync(p, 0, n * sizeof(float), st);
  const size_t blocks = (n / 4 + 255) / 256;
  const int grid = (int)(blocks < (size_t)(2 * num_sms()) ? (blocks > 0 ? blocks : 1) : 2 * num_sms());
  zero_f32_kernel<<<grid, 256, 0, st>>>(p, n);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* Y, const int32_t* inv, const float* w, int T, int k, int H, int out_dtype,
                           void* out, int32_t* dev_status, cudaStream_t st) {
  const int64_t total = (int64_t)T * (H / 4);
  if (total == 0) return cudaSuccess;
  // column ranges per token so that small batches still cover the SMs twice
  // over, each range at least one float4 column per thread (256)
  const int64_t q_per_row = H / 4;
  const int64_t cs_max = q_per_row / 256 > 0 ? q_per_row / 256 : 1;
  int64_t cs = (2 * (int64_t)num_sms() + T - 1) / T;
  cs = cs < 1 ? 1 : (cs > cs_max ? cs_max : cs);
  const int64_t blocks = (int64_t)T * cs;
  const int grid = (int)(blocks < 8 * (int64_t)num_sms() ? blocks : 8 * (int64_t)num_sms());
  return launch_pdl(combine_kernel, grid, 256, 0, st, Y, inv, w, T, k, (int64_t)H, (int)cs, out_dtype, out,
                    dev_status);
}

cudaError_t launch_mx_quantize(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes,
                               uint8_t* scales, cudaStream_t st) {
  const int64_t total = rows * mx_scale_pitch(cols);
  if (total == 0) return cudaSuccess;
  const int g = grid_for(total, 256);
  if (x_dtype == NVFP4_DT_BF16)
    return launch_pdl(mx_quantize_kernel<__nv_bfloat16>, g, 256, 0, st, static_cast<const __nv_bfloat16*>(x), rows,
                      cols, ld, codes, scales);
  return launch_pdl(mx_quantize_kernel<float>, g, 256, 0, st, static_cast<const float*>(x), rows, cols, ld, codes,
                    scales);
}

cudaError_t launch_mx_quantize_scatter(const void* x_bf16, int T, int H, int k, const int32_t* inv, uint8_t* codes,
                                       uint8_t* scales, cudaStream_t st) {
  const int64_t total = (int64_t)T * mx_scale_pitch(H);
  if (total == 0) return cudaSuccess;
  return launch_pdl(mx_quantize_scatter_kernel, grid_for(total, 256), 256, 0, st,
                    static_cast<const __nv_bfloat16*>(x_bf16), T, (int64_t)H, k, inv, codes, scales);
}

cudaError_t launch_mx_pack_scales(const uint8_t* in, int E, int N, int K, uint8_t* out, cudaStream_t st) {
  const int64_t total = (int64_t)E * N * (K / 64);
  if (total == 0) return cudaSuccess;
  mx_pack_scales_kernel<<<grid_for(total, 256), 256, 0, st>>>(in, E, N, K, out);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_requant_mx(const float* G, int R, int I, uint8_t* h_codes, uint8_t* h_scales,
                                     cudaStream_t st) {
  const int64_t total = (int64_t)R * mx_scale_pitch(I);
  if (total == 0) return cudaSuccess;
  return launch_pdl(swiglu_requant_mx_kernel, grid_for(total, 256), 256, 0, st, G, (int64_t)R, (int64_t)I, h_codes,
                    h_scales);
}

cudaError_t launch_stage_in(const void* src16, void* dst16, int64_t bytes16, const void* src4, void* dst4,
                            int64_t bytes4, cudaStream_t st) {
  const int64_t n0 = bytes16 / 16, n1 = bytes4 / 4;
  const int64_t n = n0 > n1 ? n0 : n1;
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * 4;
  if (blocks > cap) blocks = cap;
  return launch_pdl(stage_in_kernel, (int)blocks, 256, 0, st, static_cast<const uint4*>(src16),
                    static_cast<uint4*>(dst16), n0, static_cast<const uint32_t*>(src4), static_cast<uint32_t*>(dst4),
                    n1);
}

}  // namespace nvfp4moe
