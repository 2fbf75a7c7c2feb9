// Routing: group-limited top-K on sigmoid affinity + bias, gates from the raw
// affinities, and the per-expert load count ("DeepSeek-V3技术报告" digest,
// mpbf.cn, section 2.2).
//
// One warp per token. Expert e lives in lane e % 32, register e / 32. The
// selection compares 64-bit keys (order-preserving bits of s' << 32 | ~e), so
// a plain maximum picks the largest biased affinity and, among equal values,
// the lowest expert index.
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;

// Groups of exactly 32 experts (one register of every lane) with the sum of
// at most the 2 largest biased affinities: the group scores are formed by a
// warp butterfly on registers, without the shared-memory copy of s'.
__host__ __device__ __forceinline__ bool butterfly_groups(int E, int G, int gk, int npl) {
  return G > 0 && E == 32 * G && npl == G && gk <= 2;
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t k) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t other = __shfl_xor_sync(0xffffffffu, k, o);
    k = other > k ? other : k;
  }
  return k;
}

template <int NPL>
__global__ void __launch_bounds__(kWarps * 32)
    route_select_kernel(const float* __restrict__ scores, const float* __restrict__ bias, int T, int E, int G,
                        int K, int M, int gk, int* __restrict__ topk_idx, float* __restrict__ topk_gate,
                        int* __restrict__ counts) {
  extern __shared__ float sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* hist = reinterpret_cast<int*>(sh);           // [E]
  float* sp_all = sh + E;                           // [kWarps][E]
  float* sp = sp_all + warp * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();

  const int gsz = E / G;
  float b[NPL];
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = lane + 32 * j;
    b[j] = e < E ? bias[e] : 0.0f;
  }

  for (int t = blockIdx.x * kWarps + warp; t < T; t += gridDim.x * kWarps) {
    const float* srow = scores + (size_t)t * E;
    float s[NPL], v[NPL];
    const bool fly = butterfly_groups(E, G, gk, NPL);
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = lane + 32 * j;
      s[j] = e < E ? srow[e] : 0.0f;
      v[j] = __fadd_rn(s[j], b[j]);  // s' = s + b, one fp32 add
      if (!fly && e < E) sp[e] = v[j];
    }
    __syncwarp();

    unsigned gmask = 0;
    if (fly) {
      // group j = register j of all lanes: top-2 of the group by a butterfly
      // (every lane ends with every group's two largest values)
      float t1[NPL], t2[NPL];
#pragma unroll
      for (int j = 0; j < NPL; ++j) {
        t1[j] = v[j];
        t2[j] = -INFINITY;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int j = 0; j < NPL; ++j) {
          const float p1 = __shfl_xor_sync(0xffffffffu, t1[j], o);
          const float p2 = __shfl_xor_sync(0xffffffffu, t2[j], o);
          const float hi = t1[j] > p1 ? t1[j] : p1;
          const float lo = t1[j] > p1 ? p1 : t1[j];
          const float m2 = t2[j] > p2 ? t2[j] : p2;
          t2[j] = lo > m2 ? lo : m2;
          t1[j] = hi;
        }
      }
      float gsa[NPL];
#pragma unroll
      for (int j = 0; j < NPL; ++j) gsa[j] = gk == 1 ? t1[j] : __fadd_rn(t1[j], t2[j]);
      // the M best groups (ties: lower group index), computed by every lane
#pragma unroll
      for (int g = 0; g < NPL; ++g) {
        int rank = 0;
#pragma unroll
        for (int g2 = 0; g2 < NPL; ++g2) rank += (gsa[g2] > gsa[g]) || (gsa[g2] == gsa[g] && g2 < g);
        if (rank < M) gmask |= 1u << g;
      }
    } else {
      // group score: sum of the gk largest s' of the group, largest first
      float gs = -INFINITY;
      if (lane < G) {
        const float* grp = sp + lane * gsz;
        if (gk <= 4) {
          float top[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          for (int j = 0; j < gsz; ++j) {
            float x = grp[j];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              if (r < gk && x > top[r]) {
                const float tmp = top[r];
                top[r] = x;
                x = tmp;
              }
            }
          }
          gs = top[0];
          for (int r = 1; r < gk; ++r) gs = __fadd_rn(gs, top[r]);
        } else {
          // larger gk (up to the whole group, the plain node sum): take the
          // members in (value desc, index asc) order one at a time
          float last_v = INFINITY;
          int last_j = -1;
          for (int r = 0; r < gk; ++r) {
            float bv = -INFINITY;
            int bj = gsz;
            for (int j = 0; j < gsz; ++j) {
              const float x = grp[j];
              const bool after_last = x < last_v || (x == last_v && j > last_j);
              if (after_last && (x > bv || (x == bv && j < bj))) {
                bv = x;
                bj = j;
              }
            }
            gs = r == 0 ? bv : __fadd_rn(gs, bv);
            last_v = bv;
            last_j = bj;
          }
        }
      }
      // the M best groups (ties: lower group index)
      int rank = 0;
      for (int g2 = 0; g2 < G; ++g2) {
        const float o = __shfl_sync(0xffffffffu, gs, g2);
        rank += (o > gs) || (o == gs && g2 < lane);
      }
      gmask = __ballot_sync(0xffffffffu, lane < G && rank < M);
    }

    uint64_t key[NPL];
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = lane + 32 * j;
      key[j] = (e < E && ((gmask >> (e / gsz)) & 1u)) ? score_key(v[j], e) : 0ull;
    }
    // K rounds of warp arg-max
    int my_e = -1;
    float my_s = 0.0f;
    for (int k = 0; k < K; ++k) {
      uint64_t best = key[0];
#pragma unroll
      for (int j = 1; j < NPL; ++j) best = key[j] > best ? key[j] : best;
      best = warp_max_u64(best);
      const int e = (int)(~(uint32_t)best);
      const int owner = e & 31, slot = e >> 5;
      float se = 0.0f;
#pragma unroll
      for (int j = 0; j < NPL; ++j) {
        if (lane == owner && j == slot) {
          key[j] = 0ull;
          se = s[j];
        }
      }
      se = __shfl_sync(0xffffffffu, se, owner);
      if (lane == k) {
        my_e = e;
        my_s = se;
      }
    }
    // gates: raw affinity over the sum of the K chosen raw affinities
    float sum = 0.0f;
    for (int k = 0; k < K; ++k) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, my_s, k));
    if (lane < K) {
      topk_idx[(size_t)t * K + lane] = my_e;
      topk_gate[(size_t)t * K + lane] = __fdiv_rn(my_s, sum);
      atomicAdd(&hist[my_e], 1);
    }
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = hist[e];
    if (c) atomicAdd(&counts[e], c);
  }
}

// Sequence-wise balance statistic of the routing (the DeepSeek-V3 report's
// sequence-level balance loss, which the digest's section 2.2 keeps with a
// tiny weight), one block per run of seq_len tokens:
//   f_i = E / (K L) * (times expert i is chosen), P_i = (1/L) sum_t s_it / sum_j s_jt,
//   loss = alpha * sum_i f_i P_i.
// Deterministic: row sums by a fixed warp butterfly, each (phase, expert)
// thread sums its tokens in order, partials are combined in a fixed order.
constexpr int kBalThreads = 1024;
constexpr int kBalChunk = 1024;  // tokens whose row sums are staged at a time

__global__ void __launch_bounds__(kBalThreads)
    seq_balance_kernel(const float* __restrict__ scores, const int* __restrict__ topk_idx, int T, int E, int K,
                       int seq_len, float alpha, float* __restrict__ loss, float* __restrict__ f_out,
                       float* __restrict__ p_out) {
  __shared__ float rs[kBalChunk];
  __shared__ float part[kBalThreads];
  __shared__ int cnt[512];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * seq_len;
  const int L = min(seq_len, T - t0);
  const int nph = kBalThreads / E;  // token phases per expert (E <= 512)
  const int e = tid % E, ph = tid / E;
  const bool active = ph < nph;
  for (int i = tid; i < E; i += kBalThreads) cnt[i] = 0;
  __syncthreads();
  const int* idx = topk_idx + (size_t)t0 * K;
  for (int i = tid; i < L * K; i += kBalThreads) {
    const int x = idx[i];
    if (x >= 0 && x < E) atomicAdd(&cnt[x], 1);
  }
  float acc = 0.0f;
  for (int c0 = 0; c0 < L; c0 += kBalChunk) {
    const int n = min(kBalChunk, L - c0);
    for (int tt = warp; tt < n; tt += kBalThreads / 32) {
      const float* row = scores + (size_t)(t0 + c0 + tt) * E;
      float v = 0.0f;
      for (int j = lane; j < E; j += 32) v += row[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) rs[tt] = v;
    }
    __syncthreads();
    if (active)
      for (int tt = ph; tt < n; tt += nph) acc += __fdiv_rn(scores[(size_t)(t0 + c0 + tt) * E + e], rs[tt]);
    __syncthreads();
  }
  part[tid] = active ? acc : 0.0f;
  __syncthreads();
  float contrib = 0.0f;
  if (tid < E) {
    float P = 0.0f;
    for (int q = 0; q < nph; ++q) P += part[q * E + tid];
    P = __fdiv_rn(P, (float)L);
    const float f = (float)((double)E * cnt[tid] / ((double)K * L));
    if (f_out) f_out[(size_t)blockIdx.x * E + tid] = f;
    if (p_out) p_out[(size_t)blockIdx.x * E + tid] = P;
    contrib = f * P;
  }
  __syncthreads();
  part[tid] = contrib;
  __syncthreads();
  for (int w = kBalThreads / 2; w > 0; w >>= 1) {
    if (tid < w) part[tid] += part[tid + w];
    __syncthreads();
  }
  if (tid == 0) loss[blockIdx.x] = alpha * part[0];
}

}  // namespace

cudaError_t launch_seq_balance(const float* scores, const int* topk_idx, int T, int E, int K, int seq_len,
                               float alpha, float* loss, float* f, float* p, cudaStream_t st) {
  if (E > 512 || seq_len <= 0) return cudaErrorInvalidValue;
  const int n_seq = (T + seq_len - 1) / seq_len;
  if (n_seq == 0) return cudaSuccess;
  seq_balance_kernel<<<n_seq, kBalThreads, 0, st>>>(scores, topk_idx, T, E, K, seq_len, alpha, loss, f, p);
  return cudaGetLastError();
}

cudaError_t launch_route_select(const float* scores, const float* bias, int T, int E, int G, int K, int M, int gk,
                                int* topk_idx, float* topk_gate, int* counts, int num_sms, cudaStream_t st) {
  const int npl = (E + 31) / 32;
  // the histogram, and (unless the group scores come from the butterfly)
  // each warp's copy of s'
  const int npl_k = npl <= 8 ? npl : npl <= 12 ? 12 : 16;  // the instantiation that runs
  const size_t smem = (size_t)(E + (butterfly_groups(E, G, gk, npl_k) ? 0 : kWarps * E)) * sizeof(float);
  const int blocks = std::max(1, std::min((T + kWarps - 1) / kWarps, num_sms * 4));
#define MOE_ROUTE_CASE(N)                                                                         \
  case N:                                                                                         \
    route_select_kernel<N><<<blocks, kWarps * 32, smem, st>>>(scores, bias, T, E, G, K, M, gk,    \
                                                              topk_idx, topk_gate, counts);       \
    break;
  switch (npl) {
    MOE_ROUTE_CASE(1)
    MOE_ROUTE_CASE(2)
    MOE_ROUTE_CASE(3)
    MOE_ROUTE_CASE(4)
    MOE_ROUTE_CASE(5)
    MOE_ROUTE_CASE(6)
    MOE_ROUTE_CASE(7)
    MOE_ROUTE_CASE(8)
    MOE_ROUTE_CASE(12)
    MOE_ROUTE_CASE(16)
    default:
      if (npl <= 12) {
        route_select_kernel<12><<<blocks, kWarps * 32, smem, st>>>(scores, bias, T, E, G, K, M, gk, topk_idx,
                                                                   topk_gate, counts);
      } else {
        route_select_kernel<16><<<blocks, kWarps * 32, smem, st>>>(scores, bias, T, E, G, K, M, gk, topk_idx,
                                                                   topk_gate, counts);
      }
  }
#undef MOE_ROUTE_CASE
  return cudaGetLastError();
}

}  // namespace moe
