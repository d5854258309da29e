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
// Exactness: an 8-bit float has at most 4 significant bits and a magnitude
// in [2^-16, 2^16) or zero, so its fp16 and fp32 forms are exact, and so is
// the fp32 product x * 2^(e - 127) for every scale below 255: the smallest,
// 2^-143, is a multiple of fp32's subnormal step 2^-149, and a product of
// 2^128 or more is infinite in fp32 and rounds to infinity in bf16 as well.
// The cast to bf16 (round to nearest even) is therefore the one rounding:
// each value is the exact value rounded once.  NaN elements or scales give
// NaN, E5M2 infinities stay infinite, zeros keep their sign.
//
// Memory-bound: a thread converts a group of 16 consecutive bytes (one
// 16-byte load, two 16-byte stores, the group's scales in one load), two
// elements at a time through fp16 and fp32 and one packed rounding to bf16.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fgemm_internal.h"

namespace fgemm {

namespace {

// x * 2^(e - 127) rounded once to bf16, for any scale (the general path).
__device__ __forceinline__ uint16_t scaled_bf16(float x, uint8_t e) {
  if (e == 255u) return 0x7FC0u;  // NaN scale
  // 2^(e - 127) as fp32: normal for e >= 1, the subnormal 2^-127 for e = 0
  const float s = e == 0 ? __int_as_float(1 << 22) : __int_as_float(static_cast<int>(e) << 23);
  return __bfloat16_as_ushort(__float2bfloat16_rn(x * s));  // x * s is exact
}

// Bit 7 of each byte set where that byte of `s` lies outside [lo, hi]
// (lo < 128 <= hi); the other bits are junk.
__device__ __forceinline__ uint32_t bytes_outside4(uint32_t s, uint32_t lo, uint32_t hi) {
  const uint32_t ge_lo = ((s | 0x80808080u) - lo * 0x01010101u) | s;
  const uint32_t ns = ~s;
  const uint32_t le_hi = ((ns | 0x80808080u) - (255u - hi) * 0x01010101u) | ns;
  return ~(ge_lo & le_hi);
}

// One 16-column group: its 16 bytes and the scales that apply to them, both
// packed four to a word (scales along rows: only s[0], the group's one scale).
struct MxGroup {
  uint32_t w[4];
  uint32_t s[4];
};

// A job as the kernel sees it: the matrix, whether every full group's
// element, output and (down columns) scale rows are 16-byte aligned, and its
// count of 16-column groups per row.
struct MxJobDev {
  const uint8_t* X;
  const uint8_t* S;
  uint16_t* Y;
  long long ldx, lds, ldy, rows;
  int cols, groups, fmt, along, vec, svec;
};

struct MxLaunch {
  MxJobDev job[2];
};

template <int ALONG>
__device__ __forceinline__ void mx_load(const MxJobDev& j, long long r, int c0, bool whole, MxGroup& g) {
  const uint8_t* src = j.X + r * j.ldx + c0;
  if (whole) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
    g.w[0] = v.x;
    g.w[1] = v.y;
    g.w[2] = v.z;
    g.w[3] = v.w;
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      g.w[q] = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (c0 + 4 * q + i < j.cols) g.w[q] |= static_cast<uint32_t>(src[4 * q + i]) << (8 * i);
    }
  }
  if (ALONG == 0) {  // a 16-column group lies in one 32-block of its row
    g.s[0] = __ldg(j.S + r * j.lds + (c0 >> 5));
  } else {           // one scale per column, from the row of the 32-block
    const uint8_t* srow = j.S + (r >> 5) * j.lds + c0;
    if (whole && j.svec) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(srow));
      g.s[0] = v.x;
      g.s[1] = v.y;
      g.s[2] = v.z;
      g.s[3] = v.w;
    } else {
      // columns past the end get scale 127 (2^0): their elements are zero
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        g.s[q] = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t e = c0 + 4 * q + i < j.cols ? __ldg(srow + 4 * q + i) : 127u;
          g.s[q] |= e << (8 * i);
        }
      }
    }
  }
}

__device__ __forceinline__ void mx_store(uint16_t* dst, int c0, int cols, bool whole, const uint32_t (&o)[8]) {
  if (whole) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (c0 + i < cols) dst[i] = static_cast<uint16_t>(o[i >> 1] >> (16 * (i & 1)));
  }
}

// The general path, for a group with a scale of 0 or 255: one value at a
// time.  Kept out of line so that the common path stays small.
__device__ __noinline__ void mx_group_general(uint16_t* dst, int c0, int cols, bool whole, MxGroup g, int fmt,
                                              int along) {
  const __nv_fp8_interpretation_t interp = fmt == 0 ? __NV_E4M3 : __NV_E5M2;
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t x = (g.w[i >> 2] >> (8 * (i & 3))) & 0xFFu;
    const uint8_t e = static_cast<uint8_t>(along == 0 ? g.s[0] : g.s[i >> 2] >> (8 * (i & 3)));
    const float f = __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(x), interp)));
    const uint32_t v = scaled_bf16(f, e);
    if (i & 1)
      o[i >> 1] |= v << 16;
    else
      o[i >> 1] = v;
  }
  mx_store(dst, c0, cols, whole, o);
}

// One group through fp32: every 8-bit value (at most 4 significant bits) is
// exact in fp16 and fp32, and x * 2^(e - 127) is exact in fp32 for e in
// [1, 254] (the smallest product 2^-142 lies above fp32's subnormal step and
// an overflow is infinite in both fp32 and bf16), so the one rounding to bf16
// is the only one.  Zeros, infinities and NaNs pass through the multiply.
// Scales 0 and 255 take the general path.
template <int FMT, int ALONG>
__device__ __forceinline__ void mx_group(uint16_t* dst, int c0, int cols, bool whole, const MxGroup& g) {
  uint32_t bad;
  if (ALONG == 0) {
    bad = (g.s[0] - 1u > 253u) ? 1u : 0u;
  } else {
    bad = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) bad |= bytes_outside4(g.s[q], 1u, 254u);
    bad &= 0x80808080u;
  }
  if (bad) {
    mx_group_general(dst, c0, cols, whole, g, FMT, ALONG);
    return;
  }
  const __nv_fp8_interpretation_t interp = FMT == 0 ? __NV_E4M3 : __NV_E5M2;
  const float s_row = __uint_as_float(g.s[0] << 23);
  uint32_t o[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>(g.w[q] >> (16 * h));
      const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pair, interp)));
      float s0 = s_row, s1 = s_row;
      if (ALONG == 1) {
        s0 = __uint_as_float(((g.s[q] >> (16 * h)) & 0xFFu) << 23);
        s1 = __uint_as_float(((g.s[q] >> (16 * h + 8)) & 0xFFu) << 23);
      }
      const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * s0, f.y * s1);
      o[2 * q + h] = *reinterpret_cast<const uint32_t*>(&b);
    }
  }
  mx_store(dst, c0, cols, whole, o);
}

// Thread t of block (x, y, z) converts 16-column group x * 256 + t of rows
// y, y + gridDim.y, ... of job z: coalesced 16-byte loads along each row.
// along == 0: scale blocks run along a row (S[r * lds + c / 32]);
// along == 1: they run down a column (S[(r / 32) * lds + c]).
template <int FMT, int ALONG>
__device__ __forceinline__ void mx_rows(const MxJobDev& j, int gi) {
  const int c0 = gi * 16;
  const bool whole = j.vec && c0 + 16 <= j.cols;
  for (long long r = blockIdx.y; r < j.rows; r += gridDim.y) {
    MxGroup g;
    mx_load<ALONG>(j, r, c0, whole, g);
    mx_group<FMT, ALONG>(j.Y + r * j.ldy + c0, c0, j.cols, whole, g);
  }
}

__device__ __forceinline__ void mx_job(const MxJobDev& j) {
  const int gi = blockIdx.x * 256 + threadIdx.x;
  if (gi >= j.groups) return;
  switch (j.fmt * 2 + j.along) {
    case 0: mx_rows<0, 0>(j, gi); break;
    case 1: mx_rows<0, 1>(j, gi); break;
    case 2: mx_rows<1, 0>(j, gi); break;
    default: mx_rows<1, 1>(j, gi); break;
  }
}

// Six resident blocks per SM (at most 40 registers a thread) keep more loads
// in flight than the unconstrained 56-register build.  The job is picked by
// a branch rather than an index so that its fields are read at fixed
// parameter offsets.
__global__ void __launch_bounds__(256, 6) mx_dequant_kernel(const __grid_constant__ MxLaunch L) {
  if (blockIdx.z == 0)
    mx_job(L.job[0]);
  else
    mx_job(L.job[1]);
}

}  // namespace

cudaError_t launch_mx_dequant(const MxJob* jobs, int njobs, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  MxLaunch p{};
  int n = 0;
  long long max_groups = 0, max_rows = 0;
  for (int i = 0; i < njobs && i < 2; ++i) {
    const MxJob& a = jobs[i];
    if (a.rows <= 0 || a.cols <= 0) continue;
    if (a.cols > (1LL << 31) - 1) return cudaErrorInvalidValue;
    MxJobDev& d = p.job[n++];
    d.X = a.X;
    d.S = a.S;
    d.Y = a.Y;
    d.ldx = a.ldx;
    d.lds = a.lds;
    d.ldy = a.ldy;
    d.rows = a.rows;
    d.cols = static_cast<int>(a.cols);
    d.groups = static_cast<int>((a.cols + 15) / 16);
    d.fmt = a.fmt;
    d.along = a.along;
    d.vec = (reinterpret_cast<uintptr_t>(a.X) % 16 == 0) && (a.ldx % 16 == 0) &&
            (reinterpret_cast<uintptr_t>(a.Y) % 16 == 0) && (a.ldy % 8 == 0);
    d.svec = (reinterpret_cast<uintptr_t>(a.S) % 16 == 0) && (a.lds % 16 == 0);
    max_groups = d.groups > max_groups ? d.groups : max_groups;
    max_rows = a.rows > max_rows ? a.rows : max_rows;
  }
  if (n == 0) return cudaSuccess;
  // x: 256 groups per block; y: one row per block row, at most 65535
  // (row-strided beyond); z: the job
  const dim3 grid(static_cast<unsigned>((max_groups + 255) / 256),
                  static_cast<unsigned>(max_rows < 65535 ? max_rows : 65535), static_cast<unsigned>(n));
  mx_dequant_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fgemm
