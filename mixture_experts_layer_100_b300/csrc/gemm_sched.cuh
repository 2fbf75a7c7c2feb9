// Tile scheduler and epilogue helpers shared by the tcgen05 GEMM kernels.
//
// The tiles of a launch are numbered 0..total-1: first those of segment 0
// (groups with device-side row offsets, group by group), then those of
// segment 1 (one group of rows1 rows). Inside a group the m-tiles are taken
// in super-rows of kSuperRow: for each n-tile the super-row's m-tiles come
// one after the other, so that the CTAs running at the same time share the
// B panel (weights) and reuse the super-row's A panels from L2.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;          // tile rows (one TMEM lane per row)
constexpr int kSuperRow = 16;     // m-tiles walked together per n sweep
constexpr int kMaxGroups = 512;

struct Tile {
  int seg, group, m, n, row0, row_end;
};

struct Sched {
  const int* tp;    // [groups0 + 1] first tile of each group (shared memory)
  const int* mt;    // [groups0] m-tiles of each group
  const int* off;   // [groups0 + 1] row offsets
  const int* end = nullptr;  // [groups0] last row + 1 of each group's stored rows (NULL: off[g + 1])
  int groups0, tiles0, total;
  int n_tiles0, n_tiles1, mt1, rows1;
  int bm = kBM;                // rows per tile
  int super_row = kSuperRow;   // m-tiles walked together per n sweep

  __device__ __forceinline__ void raster(int local, int mt, int nt, int& m, int& n) const {
    const int sr = local / (super_row * nt);
    const int base = sr * super_row;
    const int h = min(super_row, mt - base);
    const int rem = local - sr * super_row * nt;
    n = rem / h;
    m = base + rem % h;
  }

  __device__ __forceinline__ Tile decode(int L) const {
    Tile t;
    if (L < tiles0) {
      int lo = 0, hi = groups0;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tp[mid] <= L) lo = mid; else hi = mid;
      }
      t.seg = 0;
      t.group = lo;
      raster(L - tp[lo], mt[lo], n_tiles0, t.m, t.n);
      t.row0 = off[lo] + t.m * bm;
      t.row_end = end != nullptr ? end[lo] : off[lo + 1];
    } else {
      t.seg = 1;
      t.group = 0;
      raster(L - tiles0, mt1, n_tiles1, t.m, t.n);
      t.row0 = t.m * bm;
      t.row_end = rows1;
    }
    return t;
  }
};

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * q + 0], v[8 * q + 1]);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * q + 2], v[8 * q + 3]);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * q + 4], v[8 * q + 5]);
    __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * q + 6], v[8 * q + 7]);
    w.x = *reinterpret_cast<uint32_t*>(&h0);
    w.y = *reinterpret_cast<uint32_t*>(&h1);
    w.z = *reinterpret_cast<uint32_t*>(&h2);
    w.w = *reinterpret_cast<uint32_t*>(&h3);
    d4[q] = w;
  }
}

// Bytes of shared memory one warp needs for warp_store_rows64.
constexpr int kRowStageBytes = 2048;

// Writes 64 bytes of each of a warp's 32 rows (lane r holds row r's bytes in
// w[0..3]) to base + r * pitch, passing them through a 2 KB staging block of
// shared memory so that each store instruction covers 8 rows x 64 contiguous
// bytes instead of 32 rows x 16 bytes. Staging layout: row r, 16-byte chunk j
// at r * 64 + (j ^ ((r >> 1) & 3)) * 16, conflict-free for both the row-wise
// writes and the chunk-wise reads. Rows r >= nrows are not stored. Every lane
// of the warp must call it.
__device__ __forceinline__ void warp_store_rows64(uint8_t* stg, int lane, const uint4 (&w)[4], uint8_t* base,
                                                  size_t pitch, int nrows) {
#pragma unroll
  for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16)) = w[j];
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = 8 * k + (lane >> 2), j = lane & 3;
    const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 64 + ((j ^ ((r >> 1) & 3)) * 16));
    if (r < nrows) *reinterpret_cast<uint4*>(base + (size_t)r * pitch + 16 * j) = v;
  }
  __syncwarp();
}

// The reduction form of warp_store_rows64 for fp32 rows: lane r holds 16 fp32
// values of row r in w[0..3]; they are added (red.global.add, 16 bytes at a
// time) to dst + tok(r) * pitch, where tok(r) is the `tok` value of lane r.
// The same staging block and layout make each instruction cover 8 rows x 64
// contiguous bytes. Rows r >= nrows are skipped. Every lane of the warp must
// call it.
__device__ __forceinline__ void warp_red_rows64(uint8_t* stg, int lane, const uint4 (&w)[4], float* dst, int tok,
                                                size_t pitch, int nrows) {
#pragma unroll
  for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) * 16)) = w[j];
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = 8 * k + (lane >> 2), j = lane & 3;
    const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 64 + ((j ^ ((r >> 1) & 3)) * 16));
    const int tr = __shfl_sync(0xffffffffu, tok, r);
    if (r < nrows)
      ptx::red_add_v4_f32(dst + (size_t)tr * pitch + 4 * j, __uint_as_float(v.x), __uint_as_float(v.y),
                          __uint_as_float(v.z), __uint_as_float(v.w));
  }
  __syncwarp();
}

// 32 fp32 values -> 32 bf16 (round to nearest even) packed in four 16-byte words.
__device__ __forceinline__ void pack_bf16x32(const float* v, uint4 (&w)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * q + 0], v[8 * q + 1]);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * q + 2], v[8 * q + 3]);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * q + 4], v[8 * q + 5]);
    __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * q + 6], v[8 * q + 7]);
    w[q].x = *reinterpret_cast<uint32_t*>(&h0);
    w[q].y = *reinterpret_cast<uint32_t*>(&h1);
    w[q].z = *reinterpret_cast<uint32_t*>(&h2);
    w[q].w = *reinterpret_cast<uint32_t*>(&h3);
  }
}

__device__ __forceinline__ void add_bf16x32(float* acc, const __nv_bfloat16* src, float g) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w = __ldg(s4 + q);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 f = __bfloat1622float2(h[j]);
      acc[8 * q + 2 * j + 0] = fmaf(g, f.x, acc[8 * q + 2 * j + 0]);
      acc[8 * q + 2 * j + 1] = fmaf(g, f.y, acc[8 * q + 2 * j + 1]);
    }
  }
}

}  // namespace
}  // namespace moe
