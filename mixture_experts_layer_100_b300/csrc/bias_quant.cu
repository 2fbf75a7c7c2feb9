// Auxiliary-loss-free bias update ("DeepSeek-V3技术报告" digest, mpbf.cn,
// section 2.2) and the e4m3 quantisers of the FP8 expert path (same page,
// section 3.1: FP8 GEMM inputs with per-tile scale factors).
#include "kernels.cuh"

namespace moe {
namespace {

// One block. Overloaded experts (counts_e * E > T*K) lose gamma, underloaded
// ones gain gamma; the comparison is done in 64-bit integers, the add in fp32.
__global__ void __launch_bounds__(512) bias_update_kernel(const int* __restrict__ counts, int E, long long TK,
                                                          float gamma, float* __restrict__ bias,
                                                          float* __restrict__ max_over_mean) {
  __shared__ int smax[32];
  int mx = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = counts[e];
    mx = max(mx, c);
    const long long lhs = (long long)c * E;
    if (lhs > TK) {
      bias[e] = __fsub_rn(bias[e], gamma);
    } else if (lhs < TK) {
      bias[e] = __fadd_rn(bias[e], gamma);
    }
  }
  if (max_over_mean == nullptr) return;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) smax[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    int m = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = max(m, smax[w]);
    *max_over_mean = (float)((double)m * (double)E / (double)TK);
  }
}

// 128 x 128 block quantisation of bf16 matrices [n_mat, rows, cols]. One
// block of 256 threads per 128 x 128 tile; each thread owns half a row. The
// scale follows e4m3_tile_scale (fp32 or UE8M0 rule).
__global__ void __launch_bounds__(256) quantize_blocks_kernel(const __nv_bfloat16* __restrict__ w, int rows, int cols,
                                                              uint8_t* __restrict__ q, float* __restrict__ scale,
                                                              bool ue8m0) {
  const int bc = blockIdx.x, br = blockIdx.y, mat = blockIdx.z;
  const int nbr = gridDim.y, nbc = gridDim.x;
  const int r = br * 128 + (threadIdx.x >> 1);
  const int c0 = bc * 128 + (threadIdx.x & 1) * 64;
  const __nv_bfloat16* src = w + (size_t)mat * rows * cols;
  float amax = 0.0f;
  if (r < rows) {
    for (int j = 0; j < 64; ++j) {
      const int c = c0 + j;
      if (c < cols) amax = fmaxf(amax, fabsf(__bfloat162float(src[(size_t)r * cols + c])));
    }
  }
  __shared__ float red[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
  const float s = e4m3_tile_scale(m, ue8m0);
  if (threadIdx.x == 0) scale[((size_t)mat * nbr + br) * nbc + bc] = s;
  if (r < rows) {
    uint8_t* dst = q + (size_t)mat * rows * cols;
    for (int j = 0; j < 64; ++j) {
      const int c = c0 + j;
      if (c < cols) dst[(size_t)r * cols + c] = f32_to_e4m3(__fdiv_rn(__bfloat162float(src[(size_t)r * cols + c]), s));
    }
  }
}

// 1 x 128 tiles of a bf16 activation matrix [rows, d] (d % 128 == 0): codes
// [rows, d], scales tile-major [d/128, rows]. Each warp takes two tiles per
// step, one per half-warp; the loop is uniform across the warp so that the
// shuffles always see all 32 lanes. The scale follows e4m3_tile_scale.
__global__ void __launch_bounds__(256) quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, int rows, int d,
                                                            uint8_t* __restrict__ q, float* __restrict__ scale,
                                                            bool ue8m0) {
  const int ntiles = d / 128;
  const long long total = (long long)rows * ntiles;
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; 2 * w < total; w += nwarps) {
    const long long i = 2 * w + (lane >> 4);
    const bool act = i < total;
    const int row = act ? (int)(i / ntiles) : 0, tile = act ? (int)(i % ntiles) : 0;
    float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float amax = 0.0f;
    if (act) {
      const uint4 v4 = reinterpret_cast<const uint4*>(x + (size_t)row * d + tile * 128)[lane & 15];
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v4);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 v = __bfloat1622float2(h[j]);
        f[2 * j] = v.x;
        f[2 * j + 1] = v.y;
        amax = fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y)));
      }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (!act) continue;
    const float s = e4m3_tile_scale(amax, ue8m0);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) lo |= (uint32_t)f32_to_e4m3(__fdiv_rn(f[j], s)) << (8 * j);
#pragma unroll
    for (int j = 0; j < 4; ++j) hi |= (uint32_t)f32_to_e4m3(__fdiv_rn(f[4 + j], s)) << (8 * j);
    reinterpret_cast<uint2*>(q + (size_t)row * d + tile * 128)[lane & 15] = make_uint2(lo, hi);
    if ((lane & 15) == 0) scale[(size_t)tile * rows + row] = s;
  }
}

// Rows of fp32 values split for the three-product tf32 GEMMs: row r of src
// [rows, cols] becomes dst[r] = [hi (cols) | lo (cols)], hi = tf32_hi(x),
// lo = x - hi. Four values per thread and iteration.
__global__ void __launch_bounds__(256) split_tf32_kernel(const float4* __restrict__ src, long long rows, int cols4,
                                                         float4* __restrict__ dst) {
  const long long n = rows * cols4;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / cols4;
    const int c = (int)(i - r * cols4);
    const float4 v = src[i];
    const float4 h = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
    dst[2 * r * cols4 + c] = h;
    dst[2 * r * cols4 + cols4 + c] = make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w);
  }
}

}  // namespace

cudaError_t launch_split_tf32(const float* src, long long rows, int cols, float* dst, int num_sms, cudaStream_t st) {
  const long long n = rows * (cols / 4);
  if (n == 0) return cudaSuccess;
  const int blocks = (int)std::max(1LL, std::min((n + 255) / 256, (long long)num_sms * 8));
  split_tf32_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(src), rows, cols / 4,
                                            reinterpret_cast<float4*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_bias_update(const int* counts, int E, long long TK, float gamma, float* bias,
                               float* max_over_mean, cudaStream_t st) {
  bias_update_kernel<<<1, 512, 0, st>>>(counts, E, TK, gamma, bias, max_over_mean);
  return cudaGetLastError();
}

cudaError_t launch_quantize_blocks(const __nv_bfloat16* w, int n_mat, int rows, int cols, uint8_t* q, float* scale,
                                   bool ue8m0, cudaStream_t st) {
  dim3 grid((cols + 127) / 128, (rows + 127) / 128, n_mat);
  quantize_blocks_kernel<<<grid, 256, 0, st>>>(w, rows, cols, q, scale, ue8m0);
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const __nv_bfloat16* x, int rows, int d, uint8_t* q, float* scale, bool ue8m0,
                                 int num_sms, cudaStream_t st) {
  const long long warps = ((long long)rows * (d / 128) + 1) / 2;
  const long long blocks = std::max(1LL, std::min((warps * 32 + 255) / 256, (long long)num_sms * 16));
  quantize_rows_kernel<<<(int)blocks, 256, 0, st>>>(x, rows, d, q, scale, ue8m0);
  return cudaGetLastError();
}

}  // namespace moe
