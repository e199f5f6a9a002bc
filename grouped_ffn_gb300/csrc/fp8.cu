// FP8 dispatch: quantize token rows to E4M3 on the way into the dispatched
// buffer, and restore bf16 rows on the receiving side.
//
// "Mixture-of-Experts Inference", "Communication pressure": the token
// activations can be quantized, for example to FP8, before dispatch, which
// shrinks what the all-to-all moves.  Here the dispatched buffer stands in
// for the all-to-all's payload: per row, H E4M3 bytes plus one fp32 scale per
// 128 channels instead of 2*H bf16 bytes.
//
// Scale of a (token, 128-channel) block: the power of two 2^e with the
// smallest e such that the block's largest magnitude is at most 448 (the
// largest finite E4M3 value) times 2^e, e clamped to [-126, 127], e = 0 for
// an all-zero block.  Dividing by a power of two is exact, so the only
// rounding is the conversion to E4M3 (nearest, ties to even, which the
// cvt.rn.satfinite conversion does).  Restoring multiplies the E4M3 value by
// 2^e (exact in fp32) and rounds once to bf16.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace {

constexpr int kBlock = 128;         // channels per scale
constexpr int kQuantThreads = 256;  // 16 half-warps, one 128-channel block each at a time
constexpr int kDeqThreads = 256;

// Exponent e of the block scale from the block's largest |x| as bf16 bits.
__device__ __forceinline__ int block_exponent(uint32_t amax_bits) {
  if (amax_bits == 0) return 0;
  const int field = (int)((amax_bits >> 7) & 0xFF);
  if (field == 0) return -126;  // subnormal: 448 * 2^e >= amax already at the clamp
  // amax = M * 2^q with M in [1, 2); 448 = 1.75 * 2^8, so e = q - 8, plus
  // one when M > 1.75 (mantissa bits above 0b1100000)
  const int q = field - 127;
  const int e = q - 8 + ((amax_bits & 0x7F) > 0x60 ? 1 : 0);
  return e < -126 ? -126 : (e > 127 ? 127 : e);
}

__device__ __forceinline__ float pow2f(int e) {  // e in [-126, 127]
  return __int_as_float((127 + e) << 23);
}

// One CTA per token (grid-stride).  Half-warp h of the CTA quantizes blocks
// h, h + 16, h + 32, ...: each lane converts 8 channels (one 16-byte load)
// of a block and the half-warp reduces the block maximum with shuffles.  A
// lane first loads its share of up to kPerLane blocks, so that many loads
// are in flight, then quantizes them and writes the codes of each block to
// the token's k destination rows (8 bytes a lane, 128 contiguous bytes a
// half-warp).
constexpr int kPerLane = 4;

__device__ __forceinline__ uint2 quantize8(const uint4 &v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t packed[2];
#pragma unroll
  for (int i = 0; i < 4; i += 2) {
    const float2 lo = make_float2(__uint_as_float(w[i] << 16) * inv,
                                  __uint_as_float(w[i] & 0xFFFF0000u) * inv);
    const float2 hi = make_float2(__uint_as_float(w[i + 1] << 16) * inv,
                                  __uint_as_float(w[i + 1] & 0xFFFF0000u) * inv);
    const uint32_t c0 = __nv_cvt_float2_to_fp8x2(lo, __NV_SATFINITE, __NV_E4M3);
    const uint32_t c1 = __nv_cvt_float2_to_fp8x2(hi, __NV_SATFINITE, __NV_E4M3);
    packed[i / 2] = (c0 & 0xFFFFu) | (c1 << 16);
  }
  return make_uint2(packed[0], packed[1]);
}

__device__ __forceinline__ uint32_t abs_max_bits(const uint4 &v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  return m;
}

__global__ void __launch_bounds__(kQuantThreads) permute_fp8_kernel(
    const uint4 *__restrict__ x, int64_t T, int H, int k, const int32_t *__restrict__ dest_row,
    int64_t n_rows, uint2 *__restrict__ xq, float *__restrict__ xs, int32_t *status) {
  moe::pdl_wait();
  moe::pdl_trigger();
  constexpr int kHalfWarps = kQuantThreads / 16;
  const int sub = threadIdx.x & 15;
  const int hw = threadIdx.x >> 4;
  const int nb = H / kBlock;
  const int H8 = H / 8;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const int32_t *dr = dest_row + t * k;
    for (int b0 = hw; b0 < nb; b0 += kHalfWarps * kPerLane) {
      uint4 v[kPerLane];
#pragma unroll
      for (int u = 0; u < kPerLane; ++u) {
        const int b = b0 + u * kHalfWarps;
        v[u] = b < nb ? moe::ld_stream_u4(x + t * H8 + b * 16 + sub) : make_uint4(0, 0, 0, 0);
      }
      uint32_t m[kPerLane];
#pragma unroll
      for (int u = 0; u < kPerLane; ++u) m[u] = abs_max_bits(v[u]);
#pragma unroll
      for (int off = 8; off > 0; off >>= 1)
#pragma unroll
        for (int u = 0; u < kPerLane; ++u) m[u] = max(m[u], __shfl_xor_sync(0xffffffffu, m[u], off));
      uint2 q[kPerLane];
      float scale[kPerLane];
#pragma unroll
      for (int u = 0; u < kPerLane; ++u) {
        const int e = block_exponent(m[u]);
        q[u] = quantize8(v[u], pow2f(-e));
        scale[u] = pow2f(e);
      }
      for (int j = 0; j < k; ++j) {
        const int32_t r = __ldg(dr + j);
        if (r < 0 || r >= n_rows) {  // -1: dropped by a fixed-capacity layout
          if (r != -1 && sub == 0 && b0 == hw)
            moe::report_error(status, MOE_ERR_DEVICE_INDEX, (int32_t)(t * k + j), moe::K_PERMUTE);
          continue;
        }
        uint2 *dst = xq + (int64_t)r * (H / 8) + sub;
#pragma unroll
        for (int u = 0; u < kPerLane; ++u) {
          const int b = b0 + u * kHalfWarps;
          if (b < nb) {
            dst[b * (kBlock / 8)] = q[u];
            if (sub == 0) xs[(int64_t)r * nb + b] = scale[u];
          }
        }
      }
    }
  }
}

// Grid-stride over 8-channel pieces of the dispatched rows: a lane loads 8
// codes (8 bytes) and stores 8 bf16 values (one 16-byte store), so every
// store instruction of a warp covers 512 contiguous bytes.  Each thread
// issues kDeqPerLane loads before converting.  With a fixed-capacity layout
// (masked_m != NULL) rows past a slot's used count are padding and skipped.
constexpr int kDeqPerLane = 8;

__global__ void __launch_bounds__(kDeqThreads) dequant_fp8_kernel(
    const uint2 *__restrict__ xq, const float *__restrict__ xs, int64_t n_rows, int H, int cap,
    const int32_t *__restrict__ masked_m, uint4 *__restrict__ out) {
  moe::pdl_wait();
  moe::pdl_trigger();
  const int per_row = H / 8;
  const int nb = H / kBlock;
  const int64_t total = n_rows * per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < total;
       i0 += stride * kDeqPerLane) {
    uint2 q[kDeqPerLane];
    float scale[kDeqPerLane];
    bool ok[kDeqPerLane];
#pragma unroll
    for (int u = 0; u < kDeqPerLane; ++u) {
      const int64_t i = i0 + u * stride;
      const int64_t row = i / per_row;
      ok[u] = i < total;
      if (ok[u] && masked_m != nullptr) {
        const int64_t s = row / cap;
        ok[u] = (int)(row - s * cap) < __ldg(masked_m + s);
      }
      if (ok[u]) {
        q[u] = __ldcs(xq + i);
        scale[u] = __ldg(xs + row * nb + (int)(i - row * per_row) / (kBlock / 8));
      }
    }
#pragma unroll
    for (int u = 0; u < kDeqPerLane; ++u) {
      if (!ok[u]) continue;
      const uint32_t w[2] = {q[u].x, q[u].y};
      uint32_t o[4];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[c] >> (16 * h)) & 0xFFFFu);
          const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3)));
          __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale[u], f.y * scale[u]);
          o[2 * c + h] = *reinterpret_cast<uint32_t *>(&b);
        }
      }
      out[i0 + u * stride] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

extern "C" moe_status moe_permute_fp8(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                                      const int32_t *dest_row, int64_t n_rows, uint8_t *xq,
                                      float *x_scale, void *ws, size_t ws_bytes, void *stream) {
  if (T < 0 || H < 1 || k < 1 || n_rows < 0) return MOE_ERR_INVALID_ARG;
  if (H % kBlock != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !dest_row || ((!xq || !x_scale) && n_rows > 0)) return MOE_ERR_INVALID_ARG;
  if (!moe_host::aligned16(x) || !moe_host::aligned16(xq) ||
      (reinterpret_cast<uintptr_t>(x_scale) & 3u) != 0)
    return MOE_ERR_INVALID_ARG;
  if (moe_status s = moe_host::check_ws(ws, ws_bytes, moe::kStatusBytes)) return s;
  const int64_t lim = (int64_t)moe_host::sm_count() * 8;
  const unsigned grid = (unsigned)(T < lim ? T : lim);
  return moe_host::launch_pdl(permute_fp8_kernel, dim3(grid), dim3(kQuantThreads), 0,
                              static_cast<cudaStream_t>(stream), reinterpret_cast<const uint4 *>(x),
                              T, H, k, dest_row, n_rows, reinterpret_cast<uint2 *>(xq), x_scale,
                              moe_host::status_ptr(ws));
}

extern "C" moe_status moe_dequant_fp8(const uint8_t *xq, const float *x_scale, int64_t n_rows,
                                      int32_t H, int32_t cap, const int32_t *masked_m,
                                      uint16_t *x_perm, void *ws, size_t ws_bytes, void *stream) {
  (void)ws;
  (void)ws_bytes;
  if (n_rows < 0 || H < 1) return MOE_ERR_INVALID_ARG;
  if (H % kBlock != 0) return MOE_ERR_UNSUPPORTED;
  if (masked_m && (cap < 1 || n_rows % cap != 0)) return MOE_ERR_INVALID_ARG;
  if (n_rows == 0) return MOE_OK;
  if (!xq || !x_scale || !x_perm) return MOE_ERR_INVALID_ARG;
  if (!moe_host::aligned16(xq) || !moe_host::aligned16(x_perm) ||
      (reinterpret_cast<uintptr_t>(x_scale) & 3u) != 0)
    return MOE_ERR_INVALID_ARG;
  const int64_t pieces = n_rows * (H / 8);
  int64_t blocks = (pieces + kDeqThreads - 1) / kDeqThreads;
  const int64_t lim = (int64_t)moe_host::sm_count() * 8;
  if (blocks > lim) blocks = lim;
  return moe_host::launch_pdl(dequant_fp8_kernel, dim3((unsigned)blocks), dim3(kDeqThreads), 0,
                              static_cast<cudaStream_t>(stream),
                              reinterpret_cast<const uint2 *>(xq), x_scale, n_rows, H,
                              masked_m ? cap : 1, masked_m, reinterpret_cast<uint4 *>(x_perm));
}
