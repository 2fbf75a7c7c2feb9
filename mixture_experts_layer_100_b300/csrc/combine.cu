// The combine's memory-bound passes: the per-token gate-weighted sum of the
// routed rows (gather form) and the rounding of the fp32 accumulator (scatter
// form).
#include "kernels.cuh"

namespace moe {
namespace {

// out[t] = sum_k gate[t,k] * yp[slot_pos[t,k]] when there are no shared experts.
template <typename Tv>
__global__ void gather_combine_kernel(const Tv* __restrict__ yp, const int* __restrict__ slot_pos,
                                      const float* __restrict__ gate, int T, int d, int topk, Tv* __restrict__ out) {
  const long long total = (long long)T * d;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / d), c = (int)(i % d);
    float v = 0.0f;
    for (int k = 0; k < topk; ++k) {
      const int pos = slot_pos[(size_t)t * topk + k];
      v = fmaf(gate[(size_t)t * topk + k], (float)yp[(size_t)pos * d + c], v);
    }
    out[i] = (Tv)v;
  }
}

// r[t] = sum_k gate[t,k] * yp[slot_pos[t,k]] for bf16 rows: one warp per
// token, 16-byte loads of the K routed rows (each a contiguous row of yp),
// fp32 sums, one 16-byte bf16 store per 8 columns. All K loads of a column
// chunk are issued before the first is used (KMAX >= topk, unrolled), so a
// lane keeps K requests in flight.
template <int KMAX>
__global__ void __launch_bounds__(256) routed_sum_bf16_kernel(const uint4* __restrict__ yp,
                                                              const int* __restrict__ slot_pos,
                                                              const float* __restrict__ gate, int T, int row_vecs,
                                                              int topk, uint4* __restrict__ r) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = blockIdx.x * 8 + warp; t < T; t += gridDim.x * 8) {
    int pos = 0;
    float g = 0.0f;
    if (lane < topk) {
      pos = slot_pos[(size_t)t * topk + lane];
      g = gate[(size_t)t * topk + lane];
    }
    int pk[KMAX];
    float gk[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      pk[k] = __shfl_sync(0xffffffffu, pos, k);
      gk[k] = __shfl_sync(0xffffffffu, g, k);
    }
    for (int i = lane; i < row_vecs; i += 32) {
      uint4 w[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (k < topk) w[k] = __ldg(yp + (size_t)pk[k] * row_vecs + i);
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k < topk) {
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w[k]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(h[j]);
            acc[2 * j] = fmaf(gk[k], f.x, acc[2 * j]);
            acc[2 * j + 1] = fmaf(gk[k], f.y, acc[2 * j + 1]);
          }
        }
      }
      uint4 o;
      __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[0], acc[1]);
      __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[2], acc[3]);
      __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[4], acc[5]);
      __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[6], acc[7]);
      o.x = *reinterpret_cast<uint32_t*>(&b0);
      o.y = *reinterpret_cast<uint32_t*>(&b1);
      o.z = *reinterpret_cast<uint32_t*>(&b2);
      o.w = *reinterpret_cast<uint32_t*>(&b3);
      r[(size_t)t * row_vecs + i] = o;
    }
  }
}

// out = bf16(acc), 8 values per thread and iteration (two 16-byte loads, one
// 16-byte store).
__global__ void __launch_bounds__(256) acc_to_bf16_kernel(const float4* __restrict__ acc, size_t n8,
                                                          uint4* __restrict__ out) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = __ldcs(acc + 2 * i), b = __ldcs(acc + 2 * i + 1);
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(a.x, a.y), h1 = __floats2bfloat162_rn(a.z, a.w);
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(b.x, b.y), h3 = __floats2bfloat162_rn(b.z, b.w);
    uint4 o;
    o.x = *reinterpret_cast<const uint32_t*>(&h0);
    o.y = *reinterpret_cast<const uint32_t*>(&h1);
    o.z = *reinterpret_cast<const uint32_t*>(&h2);
    o.w = *reinterpret_cast<const uint32_t*>(&h3);
    out[i] = o;
  }
}

}  // namespace

cudaError_t launch_acc_to_bf16(const float* acc, size_t n, void* out, int num_sms, cudaStream_t st) {
  const size_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  const int blocks = (int)std::max<size_t>(1, std::min<size_t>((n8 + 255) / 256, (size_t)num_sms * 8));
  acc_to_bf16_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(acc), n8, static_cast<uint4*>(out));
  return cudaGetLastError();
}

cudaError_t launch_routed_sum_bf16(const void* yp, const int* slot_pos, const float* gate, int T, int d, int topk,
                                   void* r, int num_sms, cudaStream_t st) {
  const int blocks = std::max(1, std::min((T + 7) / 8, num_sms * 16));
  const uint4* y = static_cast<const uint4*>(yp);
  uint4* o = static_cast<uint4*>(r);
  if (topk <= 8) {
    routed_sum_bf16_kernel<8><<<blocks, 256, 0, st>>>(y, slot_pos, gate, T, d / 8, topk, o);
  } else if (topk <= 16) {
    routed_sum_bf16_kernel<16><<<blocks, 256, 0, st>>>(y, slot_pos, gate, T, d / 8, topk, o);
  } else {
    routed_sum_bf16_kernel<32><<<blocks, 256, 0, st>>>(y, slot_pos, gate, T, d / 8, topk, o);
  }
  return cudaGetLastError();
}

cudaError_t launch_gather_combine(const void* yp, const int* slot_pos, const float* gate, int T, int d, int topk,
                                  bool bf16, void* out, int num_sms, cudaStream_t st) {
  const long long total = (long long)T * d;
  const int blocks = (int)std::max(1LL, std::min((total + 255) / 256, (long long)num_sms * 16));
  if (bf16) {
    gather_combine_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(yp), slot_pos,
                                                                  gate, T, d, topk,
                                                                  static_cast<__nv_bfloat16*>(out));
  } else {
    gather_combine_kernel<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(yp), slot_pos, gate, T, d, topk,
                                                         static_cast<float*>(out));
  }
  return cudaGetLastError();
}

}  // namespace moe
