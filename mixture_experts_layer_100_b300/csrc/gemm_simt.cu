// fp32 expert GEMMs on the CUDA cores (FFMA), for layers whose activations
// and weights are fp32: the output tolerance of such a layer (1e-5 of the
// largest output) is below what TF32 tensor-core inputs can deliver, so these
// shapes stay on plain fp32 arithmetic. 64 x 64 output tiles, K staged through
// shared memory in steps of 16, 4 x 4 outputs per thread.
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kT = 64;
constexpr int kK = 16;

__device__ __forceinline__ float load_b(const SimtParams& p, int g, int n, int k, int up) {
  if (p.mode == kSimtSwiGLU) {
    // out column n of the gate (up = 0) or up (up = 1) projection
    int e = g, nn = n;
    if (p.shared) {
      e = n / p.I;
      nn = n % p.I;
    }
    return p.B[((size_t)e * 2 * p.I + (size_t)up * p.I + nn) * p.Kdim + k];
  }
  int e = g, kk = k;
  if (p.shared) {
    e = k / p.I;
    kk = k % p.I;
  }
  return p.B[((size_t)e * p.N + n) * p.I + kk];
}

__global__ void __launch_bounds__(256) simt_gemm_kernel(const SimtParams p) {
  __shared__ float As[kT][kK + 1];
  __shared__ float Bg[kT][kK + 1];
  __shared__ float Bu[kT][kK + 1];
  __shared__ int s_info[3];  // group, row0, row_end
  if (threadIdx.x == 0) {
    int mi = blockIdx.y, g = -1, row0 = 0, row_end = 0;
    if (p.groups > 0) {
      for (int e = 0; e < p.groups; ++e) {
        const int o0 = p.offsets[e], o1 = p.offsets[e + 1];
        const int mt = (o1 - o0 + kT - 1) / kT;
        if (mi < mt) {
          g = e;
          row0 = o0 + mi * kT;
          row_end = o1;
          break;
        }
        mi -= mt;
      }
    } else if (mi * kT < p.rows) {
      g = 0;
      row0 = mi * kT;
      row_end = p.rows;
    }
    s_info[0] = g;
    s_info[1] = row0;
    s_info[2] = row_end;
  }
  __syncthreads();
  const int g = s_info[0], row0 = s_info[1], row_end = s_info[2];
  if (g < 0) return;
  const int n0 = blockIdx.x * kT;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16 threads, 4 x 4 each
  const bool swiglu = p.mode == kSimtSwiGLU;
  float ag[4][4] = {}, au[4][4] = {};
  for (int k0 = 0; k0 < p.Kdim; k0 += kK) {
    for (int i = threadIdx.x; i < kT * kK; i += 256) {
      const int r = i / kK, c = i % kK;
      const int row = row0 + r, k = k0 + c, n = n0 + r;
      As[r][c] = (row < row_end && k < p.Kdim) ? p.A[(size_t)row * p.lda + k] : 0.0f;
      const bool okb = n < p.N && k < p.Kdim;
      Bg[r][c] = okb ? load_b(p, g, n, k, 0) : 0.0f;
      if (swiglu) Bu[r][c] = okb ? load_b(p, g, n, k, 1) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kK; ++k) {
      float a[4], bg[4], bu[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[ty * 4 + i][k];
        bg[i] = Bg[tx * 4 + i][k];
        bu[i] = swiglu ? Bu[tx * 4 + i][k] : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ag[i][j] = fmaf(a[i], bg[j], ag[i][j]);
          au[i][j] = fmaf(a[i], bu[j], au[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = row0 + ty * 4 + i;
    if (row >= row_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= p.N) continue;
      float v = ag[i][j];
      if (swiglu) {
        v = silu(v) * au[i][j];
      } else if (p.mode == kSimtCombine) {
        for (int k = 0; k < p.topk; ++k) {
          const int pos = p.slot_pos[(size_t)row * p.topk + k];
          v = fmaf(p.gate[(size_t)row * p.topk + k], p.yp[(size_t)pos * p.N + n], v);
        }
      }
      p.out[(size_t)row * p.ldo + n] = v;
    }
  }
}

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

}  // namespace

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

cudaError_t launch_simt_gemm(const SimtParams& p, int max_mtiles, cudaStream_t st) {
  if (max_mtiles <= 0) return cudaSuccess;
  dim3 grid((p.N + kT - 1) / kT, max_mtiles);
  simt_gemm_kernel<<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

int simt_max_mtiles(int rows_total, int groups) { return (rows_total + kT - 1) / kT + groups; }

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
