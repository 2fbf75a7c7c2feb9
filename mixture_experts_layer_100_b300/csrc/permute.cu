// Expert-major permutation of the (token, slot) pairs and the row gather:
// the single-GPU stand-in for the all-to-all dispatch of the DeepSeek-V3
// pages ("DeepSeek-V3技术报告" digest, mpbf.cn, section 3.3). Every pair keeps
// its place (no dropping, section 2.2); positions are expert-major and, inside
// an expert, token-ascending.
//
// Three passes, no host synchronisation and no atomics on positions:
//   rank    one warp per chunk of 32 tokens: per-chunk histogram and, for
//           every pair, its rank among the earlier pairs of the chunk with
//           the same expert (__match_any_sync over the pairs in order);
//   scan    one warp per expert: exclusive scan of that expert's chunk
//           histogram, offset by the expert's start (a sum over counts[]);
//   scatter one warp per token: position = base[e][chunk] + rank; writes
//           slot_pos / sorted_tok and copies the token row to its K places
//           with 16-byte vector accesses (optionally quantising it to e4m3).
// Optionally (pad > 1) every expert's rows start at a multiple of pad and
// the scatter zeroes the unused rows after them, so that the expert GEMMs'
// last tile of each expert multiplies zeros instead of the next expert's
// rows (the same instructions; zero operands draw less power).
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kChunk = 32;  // tokens per rank chunk (one warp)
constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
    permute_rank_kernel(const int* __restrict__ topk_idx, int T, int K, int E, int nchunks,
                        int* __restrict__ local_rank, int* __restrict__ chunk_hist, int* err) {
  extern __shared__ int hist_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* hist = hist_all + warp * E;
  const int c = blockIdx.x * kWarps + warp;
  for (int e = lane; e < E; e += 32) hist[e] = 0;
  __syncwarp();
  if (c < nchunks) {
    const int t0 = c * kChunk;
    const int ntok = min(kChunk, T - t0);
    const int npairs = ntok * K;
    const int* src = topk_idx + (size_t)t0 * K;
    int* dst = local_rank + (size_t)t0 * K;
    for (int base = 0; base < npairs; base += 32) {
      const int q = base + lane;
      int e = q < npairs ? src[q] : -1;
      if (e >= E || e < -1 || (q < npairs && e < 0)) {
        set_error(err, kDevBadExpertIndex);
        e = -1;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int before = __popc(peers & ((1u << lane) - 1u));
      int r = 0;
      if (e >= 0) r = hist[e] + before;
      __syncwarp();
      if (e >= 0 && before == 0) hist[e] += __popc(peers);
      __syncwarp();
      if (q < npairs) dst[q] = r;
    }
    __syncwarp();
    for (int e = lane; e < E; e += 32) chunk_hist[(size_t)e * nchunks + c] = hist[e];
  }
}

__global__ void __launch_bounds__(kWarps * 32)
    permute_scan_kernel(const int* __restrict__ counts, const int* __restrict__ chunk_hist, int E, int nchunks,
                        int* __restrict__ chunk_base, int* __restrict__ offsets, int* err, int pad) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kWarps + warp;
  if (e >= E) return;
  int start = 0;  // rows of the experts before e, each rounded up to pad
  for (int j = lane; j < e; j += 32) start += (counts[j] + pad - 1) / pad * pad;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) start += __shfl_xor_sync(0xffffffffu, start, o);
  const int* h = chunk_hist + (size_t)e * nchunks;
  int* out = chunk_base + (size_t)e * nchunks;
  int carry = start;
  for (int c0 = 0; c0 < nchunks; c0 += 32) {
    const int c = c0 + lane;
    const int v = c < nchunks ? h[c] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (c < nchunks) out[c] = carry + incl - v;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    if (carry - start != counts[e]) set_error(err, kDevCountMismatch);
    offsets[e] = start;
    if (e == E - 1) offsets[E] = start + (counts[e] + pad - 1) / pad * pad;
  }
}

template <typename VecT>
__global__ void __launch_bounds__(kWarps * 32)
    permute_scatter_kernel(const int* __restrict__ topk_idx, const int* __restrict__ local_rank,
                           const int* __restrict__ chunk_base, int T, int K, int E, int nchunks,
                           const VecT* __restrict__ x, int row_vecs, int* __restrict__ sorted_tok,
                           int* __restrict__ slot_pos, VecT* __restrict__ xp, const float* __restrict__ gate_in,
                           float* __restrict__ gate_p, int pad, const int* __restrict__ offsets,
                           const int* __restrict__ counts) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (pad > 1) {
    // the unused rows of the padded layout: item (e, j) is row
    // offsets[e] + counts[e] + j when that is before offsets[e + 1]
    const VecT zero = {};
    for (int i = blockIdx.x * kWarps + warp; i < E * pad; i += gridDim.x * kWarps) {
      const int e = i / pad;
      const int row = offsets[e] + counts[e] + i % pad;
      if (row < offsets[e + 1]) {
        VecT* dst = xp + (size_t)row * row_vecs;
        for (int v = lane; v < row_vecs; v += 32) dst[v] = zero;
      }
    }
  }
  for (int t = blockIdx.x * kWarps + warp; t < T; t += gridDim.x * kWarps) {
    int pos = 0;
    if (lane < K) {
      const int e = topk_idx[(size_t)t * K + lane];
      if (e >= 0 && e < E) {
        pos = chunk_base[(size_t)e * nchunks + t / kChunk] + local_rank[(size_t)t * K + lane];
        slot_pos[(size_t)t * K + lane] = pos;
        sorted_tok[pos] = t;
        if (gate_p != nullptr) gate_p[pos] = gate_in[(size_t)t * K + lane];
      } else {
        pos = -1;
      }
    }
    const VecT* src = x + (size_t)t * row_vecs;
    if (K <= 8) {
      // positions fetched once per token; four loads per lane in flight
      // before their stores (the copy is bound by bytes in flight)
      int pk[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) pk[k] = __shfl_sync(0xffffffffu, pos, k);
      for (int i0 = lane; i0 < row_vecs; i0 += 4 * 32) {
        VecT v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (i0 + 32 * u < row_vecs) v[u] = src[i0 + 32 * u];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (k < K && pk[k] >= 0) {
            VecT* dst = xp + (size_t)pk[k] * row_vecs;
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (i0 + 32 * u < row_vecs) dst[i0 + 32 * u] = v[u];
          }
        }
      }
    } else {
      for (int i = lane; i < row_vecs; i += 32) {
        const VecT val = src[i];
        for (int k = 0; k < K; ++k) {
          const int pk = __shfl_sync(0xffffffffu, pos, k);
          if (pk >= 0) xp[(size_t)pk * row_vecs + i] = val;
        }
      }
    }
  }
}

// Same positions; each token row (bf16) is cut into 1x128 tiles and written
// to its K places as e4m3 codes, with one fp32 scale per tile:
// scale = e4m3_tile_scale(amax) (amax / 448, or the UE8M0 power of two; 1 for
// an all-zero tile), code = e4m3(v / scale).
// A half-warp covers one 128-element tile (8 elements per lane). When xq is
// given, the quantised row is also written once in token order (for the
// shared experts). The scales go out once per token, token-major
// (tok_scale[t * ntiles + tile]); scale_tiles_kernel then lays them out
// tile-major for the permuted rows, which keeps this kernel's writes whole
// sectors instead of one 4-byte store per (token, copy, tile).
__global__ void __launch_bounds__(kWarps * 32)
    permute_scatter_e4m3_kernel(const int* __restrict__ topk_idx, const int* __restrict__ local_rank,
                                const int* __restrict__ chunk_base, int T, int K, int E, int nchunks,
                                const __nv_bfloat16* __restrict__ x, int d, int* __restrict__ sorted_tok,
                                int* __restrict__ slot_pos, uint8_t* __restrict__ xp, float* __restrict__ tok_scale,
                                uint8_t* __restrict__ xq, bool ue8m0, const float* __restrict__ gate_in,
                                float* __restrict__ gate_p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = d / 128;
  for (int t = blockIdx.x * kWarps + warp; t < T; t += gridDim.x * kWarps) {
    int pos = -1;
    if (lane < K) {
      const int e = topk_idx[(size_t)t * K + lane];
      if (e >= 0 && e < E) {
        pos = chunk_base[(size_t)e * nchunks + t / kChunk] + local_rank[(size_t)t * K + lane];
        slot_pos[(size_t)t * K + lane] = pos;
        sorted_tok[pos] = t;
        if (gate_p != nullptr) gate_p[pos] = gate_in[(size_t)t * K + lane];
      }
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    // the K positions fetched once per token (K <= 8)
    int pks[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) pks[k] = __shfl_sync(0xffffffffu, pos, k);
    // four tiles per warp iteration, both loads issued first: lanes 0..15
    // take tiles 4i and 4i+2, lanes 16..31 tiles 4i+1 and 4i+3
    for (int tile00 = 0; tile00 < ntiles; tile00 += 4) {
      uint4 wv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int tl = tile00 + 2 * u + (lane >> 4);
        if (tl < ntiles) wv[u] = src[tl * 16 + (lane & 15)];
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int tile0 = tile00 + 2 * u;
        const int tile = tile0 + (lane >> 4);
        const bool act = tile < ntiles;
        float f[8];
        float amax = 0.0f;
        if (act) {
          const uint4 w = wv[u];
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 v = __bfloat1622float2(h[j]);
            f[2 * j] = v.x;
            f[2 * j + 1] = v.y;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float scale = e4m3_tile_scale(amax, ue8m0);
        uint2 packed = make_uint2(0, 0);
        if (act) {
          uint32_t lo = 0, hi = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) lo |= (uint32_t)f32_to_e4m3(__fdiv_rn(f[j], scale)) << (8 * j);
#pragma unroll
          for (int j = 0; j < 4; ++j) hi |= (uint32_t)f32_to_e4m3(__fdiv_rn(f[4 + j], scale)) << (8 * j);
          packed = make_uint2(lo, hi);
        }
        if (K <= 8) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (k < K && act && pks[k] >= 0)
              reinterpret_cast<uint2*>(xp + (size_t)pks[k] * d + tile * 128)[lane & 15] = packed;
        } else {
          for (int k = 0; k < K; ++k) {
            const int pk = __shfl_sync(0xffffffffu, pos, k);
            if (act && pk >= 0) reinterpret_cast<uint2*>(xp + (size_t)pk * d + tile * 128)[lane & 15] = packed;
          }
        }
        if (act && (lane & 15) == 0) tok_scale[(size_t)t * ntiles + tile] = scale;
        if (act && xq != nullptr) reinterpret_cast<uint2*>(xq + (size_t)t * d + tile * 128)[lane & 15] = packed;
      }
    }
  }
}

// Tile-major scales of the permuted rows, xp_scale[tile * TK + pos] =
// tok_scale[sorted_tok[pos] * ntiles + tile], and (when xq_scale is given)
// of the token-order rows, xq_scale[tile * T + t] = tok_scale[t * ntiles +
// tile]: coalesced writes, gathered reads of the small token-major table.
__global__ void __launch_bounds__(256)
    scale_tiles_kernel(const float* __restrict__ tok_scale, const int* __restrict__ sorted_tok, int T, int TK,
                       int ntiles, float* __restrict__ xp_scale, float* __restrict__ xq_scale) {
  const long long n_p = (long long)ntiles * TK;
  const long long n_q = xq_scale != nullptr ? (long long)ntiles * T : 0;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_p + n_q; i += stride) {
    if (i < n_p) {
      const int tile = (int)(i / TK), pos = (int)(i % TK);
      const int t = sorted_tok[pos];
      xp_scale[i] = (t >= 0 && t < T) ? tok_scale[(size_t)t * ntiles + tile] : 1.0f;
    } else {
      const long long j = i - n_p;
      const int tile = (int)(j / T), t = (int)(j % T);
      xq_scale[j] = tok_scale[(size_t)t * ntiles + tile];
    }
  }
}

// Row moves by an index list (the receive-side reorder of expert-parallel
// dispatch and its inverse): one warp per row, 16-byte (or 4-byte) vectors.
// gather: dst[i] = src[idx[i]]; scatter: dst[idx[i]] = src[i]. An index
// outside [0, n_other) is skipped and reported in err.
template <typename VecT, bool GATHER>
__global__ void __launch_bounds__(kWarps * 32)
    move_rows_kernel(const VecT* __restrict__ src, const int* __restrict__ idx, int n, int n_other, int row_vecs,
                     VecT* __restrict__ dst, int* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = blockIdx.x * kWarps + warp; i < n; i += gridDim.x * kWarps) {
    const int j = idx[i];
    if (j < 0 || j >= n_other) {
      if (lane == 0) set_error(err, kDevBadRowIndex);
      continue;
    }
    const VecT* s = src + (size_t)(GATHER ? j : i) * row_vecs;
    VecT* d = dst + (size_t)(GATHER ? i : j) * row_vecs;
    for (int c = lane; c < row_vecs; c += 32) d[c] = s[c];
  }
}

}  // namespace

cudaError_t launch_move_rows(const void* src, const int* idx, int n, int n_other, size_t row_bytes, void* dst,
                             bool gather, int* err, int num_sms, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int blocks = std::max(1, std::min((n + kWarps - 1) / kWarps, num_sms * 8));
  if (row_bytes % 16 == 0) {
    const int rv = (int)(row_bytes / 16);
    auto s = static_cast<const uint4*>(src);
    auto d = static_cast<uint4*>(dst);
    if (gather) {
      move_rows_kernel<uint4, true><<<blocks, kWarps * 32, 0, st>>>(s, idx, n, n_other, rv, d, err);
    } else {
      move_rows_kernel<uint4, false><<<blocks, kWarps * 32, 0, st>>>(s, idx, n, n_other, rv, d, err);
    }
  } else {
    const int rv = (int)(row_bytes / 4);
    auto s = static_cast<const uint32_t*>(src);
    auto d = static_cast<uint32_t*>(dst);
    if (gather) {
      move_rows_kernel<uint32_t, true><<<blocks, kWarps * 32, 0, st>>>(s, idx, n, n_other, rv, d, err);
    } else {
      move_rows_kernel<uint32_t, false><<<blocks, kWarps * 32, 0, st>>>(s, idx, n, n_other, rv, d, err);
    }
  }
  return cudaGetLastError();
}

int permute_chunks(int T) { return (T + kChunk - 1) / kChunk; }

cudaError_t launch_permute_rank(const int* topk_idx, int T, int K, int E, int* local_rank, int* chunk_hist, int* err,
                                cudaStream_t st) {
  const int nchunks = permute_chunks(T);
  const int blocks = (nchunks + kWarps - 1) / kWarps;
  permute_rank_kernel<<<blocks, kWarps * 32, (size_t)kWarps * E * sizeof(int), st>>>(topk_idx, T, K, E, nchunks,
                                                                                      local_rank, chunk_hist, err);
  return cudaGetLastError();
}

cudaError_t launch_permute_scan(const int* counts, const int* chunk_hist, int T, int E, int* chunk_base, int* offsets,
                                int* err, cudaStream_t st, int pad) {
  const int nchunks = permute_chunks(T);
  permute_scan_kernel<<<(E + kWarps - 1) / kWarps, kWarps * 32, 0, st>>>(counts, chunk_hist, E, nchunks, chunk_base,
                                                                         offsets, err, pad);
  return cudaGetLastError();
}

cudaError_t launch_permute_scatter(const int* topk_idx, const int* local_rank, const int* chunk_base, int T, int K,
                                   int E, const void* x, size_t row_bytes, int* sorted_tok, int* slot_pos, void* xp,
                                   int num_sms, cudaStream_t st, const float* gate_in, float* gate_p, int pad,
                                   const int* offsets, const int* counts) {
  const int nchunks = permute_chunks(T);
  const int blocks = std::max(1, std::min((T + kWarps - 1) / kWarps, num_sms * 8));
  if (pad > 1 && (offsets == nullptr || counts == nullptr)) return cudaErrorInvalidValue;
  if (row_bytes % 16 == 0) {
    permute_scatter_kernel<uint4><<<blocks, kWarps * 32, 0, st>>>(
        topk_idx, local_rank, chunk_base, T, K, E, nchunks, static_cast<const uint4*>(x), (int)(row_bytes / 16),
        sorted_tok, slot_pos, static_cast<uint4*>(xp), gate_in, gate_p, pad, offsets, counts);
  } else {
    permute_scatter_kernel<uint32_t><<<blocks, kWarps * 32, 0, st>>>(
        topk_idx, local_rank, chunk_base, T, K, E, nchunks, static_cast<const uint32_t*>(x), (int)(row_bytes / 4),
        sorted_tok, slot_pos, static_cast<uint32_t*>(xp), gate_in, gate_p, pad, offsets, counts);
  }
  return cudaGetLastError();
}

cudaError_t launch_permute_scatter_e4m3(const int* topk_idx, const int* local_rank, const int* chunk_base, int T,
                                        int K, int E, const __nv_bfloat16* x, int d, int* sorted_tok, int* slot_pos,
                                        uint8_t* xp, float* xp_scale, uint8_t* xq, float* xq_scale, float* tok_scale,
                                        bool ue8m0, int num_sms, cudaStream_t st, const float* gate_in,
                                        float* gate_p) {
  const int nchunks = permute_chunks(T);
  const int blocks = std::max(1, std::min((T + kWarps - 1) / kWarps, num_sms * 8));
  permute_scatter_e4m3_kernel<<<blocks, kWarps * 32, 0, st>>>(topk_idx, local_rank, chunk_base, T, K, E, nchunks, x,
                                                              d, sorted_tok, slot_pos, xp, tok_scale, xq, ue8m0,
                                                              gate_in, gate_p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int ntiles = d / 128;
  const long long n = (long long)ntiles * ((long long)T * K + (xq_scale != nullptr ? T : 0));
  const int sblocks = (int)std::max(1LL, std::min((n + 255) / 256, (long long)num_sms * 8));
  scale_tiles_kernel<<<sblocks, 256, 0, st>>>(tok_scale, sorted_tok, T, T * K, ntiles, xp_scale, xq_scale);
  return cudaGetLastError();
}

}  // namespace moe
