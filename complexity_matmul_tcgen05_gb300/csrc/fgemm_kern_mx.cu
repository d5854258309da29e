// fgemm_kern_mx.cu -- block-scaled 8-bit (MX) inputs to bf16.
//
// CS336 Lecture 05 notes, "Page 27. Frontiers in low precision - FP8 and
// MXFP8": elements are E4M3 or E5M2 8-bit floats, and each block of 32
// consecutive values along the reduction direction shares one E8M0 scale
// (2^(e - 127), e = 255 is NaN).  "Page 28. MXFP8 training in practice": a
// quantize / dequantize step sits in front of the matmul.  This kernel is
// that step: it writes every value x * 2^(e - 127) as bf16, which the bf16
// tensor-core GEMM then consumes.
//
// Exactness: an 8-bit float has at most 4 significant bits, so while
// x * 2^(e - 127) stays in bf16's normal range the fp32 product and its bf16
// cast are exact.  Outside it (a subnormal or an overflowing result) the
// product is formed in double precision and rounded to bf16 once
// (round-to-nearest-even), so the value equals the exact value rounded once.
// NaN elements or scales give NaN; E5M2 infinities stay infinite.
//
// Memory-bound: each thread converts 16 consecutive bytes of a row (one
// 16-byte load, two 16-byte stores), grid-strided over the matrix.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fgemm_internal.h"

namespace fgemm {

namespace {

__device__ __forceinline__ float fp8_to_float(uint8_t x, int fmt) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(x),
                                               fmt == 0 ? __NV_E4M3 : __NV_E5M2);
  return __half2float(__half(h));
}

// x * 2^(e - 127) rounded once to bf16.
__device__ __forceinline__ uint16_t scaled_bf16(float x, uint8_t e) {
  if (e == 255u) return 0x7FC0u;  // NaN scale
  // 2^(e - 127) as fp32 (normal for e >= 1, the subnormal 2^-127 for e = 0)
  const float s = e == 0 ? __int_as_float(1 << 22) : __int_as_float(static_cast<int>(e) << 23);
  const float f = x * s;
  const float af = fabsf(f);
  if (x == 0.0f || (af >= 1.1754943508222875e-38f && af <= 3.3895313892515355e+38f) || !isfinite(x)) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));  // exact: at most 4 significant bits
  }
  // subnormal or overflowing result: the exact product, rounded once
  const double d = static_cast<double>(x) * __longlong_as_double(static_cast<long long>(e - 127 + 1023) << 52);
  return __bfloat16_as_ushort(__double2bfloat16(d));
}

// along == 0: scale blocks run along a row (S[r * lds + c / 32]);
// along == 1: they run down a column (S[(r / 32) * lds + c]).
__global__ void __launch_bounds__(256) mx_dequant_kernel(const uint8_t* __restrict__ X, long long ldx,
                                                         const uint8_t* __restrict__ S, long long lds,
                                                         int fmt, int along, long long rows,
                                                         long long cols, uint16_t* __restrict__ Y,
                                                         long long ldy) {
  const long long groups_per_row = (cols + 15) / 16;
  const long long total = rows * groups_per_row;
  for (long long g = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = g / groups_per_row;
    const long long c0 = (g - r * groups_per_row) * 16;
    const uint8_t* src = X + r * ldx + c0;
    uint16_t* dst = Y + r * ldy + c0;
    const bool whole = c0 + 16 <= cols && ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) &&
                       ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0);
    uint8_t b[16];
    if (whole) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 16; ++i) b[i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) b[i] = c0 + i < cols ? src[i] : 0;
    }
    uint16_t o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const long long c = c0 + i;
      const uint8_t e = along == 0 ? S[r * lds + (c >> 5)] : S[(r >> 5) * lds + c];
      o[i] = c < cols ? scaled_bf16(fp8_to_float(b[i], fmt), e) : 0;
    }
    if (whole) {
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      d4[0] = make_uint4(o[0] | (static_cast<uint32_t>(o[1]) << 16), o[2] | (static_cast<uint32_t>(o[3]) << 16),
                         o[4] | (static_cast<uint32_t>(o[5]) << 16), o[6] | (static_cast<uint32_t>(o[7]) << 16));
      d4[1] = make_uint4(o[8] | (static_cast<uint32_t>(o[9]) << 16), o[10] | (static_cast<uint32_t>(o[11]) << 16),
                         o[12] | (static_cast<uint32_t>(o[13]) << 16), o[14] | (static_cast<uint32_t>(o[15]) << 16));
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (c0 + i < cols) dst[i] = o[i];
    }
  }
}

}  // namespace

cudaError_t launch_mx_dequant(const uint8_t* X, long long ldx, const uint8_t* S, long long lds, int fmt,
                              int along, long long rows, long long cols, uint16_t* Y, long long ldy,
                              int num_sms, cudaStream_t stream) {
  const long long groups = rows * ((cols + 15) / 16);
  if (groups == 0) return cudaSuccess;
  // a few waves of resident blocks (8 x 256 threads per SM), grid-strided
  const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 1) * 8 * 4;
  const long long want = (groups + 255) / 256;
  const int grid = static_cast<int>(want < cap ? want : cap);
  mx_dequant_kernel<<<grid, 256, 0, stream>>>(X, ldx, S, lds, fmt, along, rows, cols, Y, ldy);
  return cudaGetLastError();
}

}  // namespace fgemm
