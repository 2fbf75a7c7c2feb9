// FP8 (e4m3) persistent grouped GEMM on tcgen05 with per-tile scales and
// fp32 promotion ("DeepSeek-V3技术报告" digest, mpbf.cn, section 3.1: FP8 GEMM
// inputs, scale factors per small tile, higher-precision accumulation).
//
// Operands: A rows in 1x128 e4m3 tiles with one fp32 scale per (row, tile),
// stored tile-major [K/128, rows]; B (weights) in 128x128 e4m3 blocks with
// one fp32 scale per block, [groups, N/128, K/128]. Each 128-wide K block is
// multiplied on the tensor cores into one of two TMEM buffers (a fresh
// accumulation per block); the epilogue warps drain the buffer, multiply the
// partial sums by scale_a(row, kb) * scale_b(n-block, kb) and add them into
// fp32 registers, so the scaled sum over K blocks is formed outside the
// tensor core at full fp32 precision while the next block is multiplied.
//
// Roles: warp 0 TMA producer, warp 1 MMA issuer, then the epilogue warps;
// epilogue warp w drains TMEM lane quarter w % 4. GEMM1 (SwiGLU, 320
// threads): 8 epilogue warps, column half (w - 2) / 4 (128 of the tile's 256
// columns), 128 fp32 accumulators each. Down projections (576 threads): 16
// epilogue warps, column slice (w - 2) / 4 (64 columns), 64 accumulators
// each, loaded 16 columns at a time to fit 96 registers: the drain of a K
// block is spread over twice the warps, which pays for their short K (a
// quarter of GEMM1's blocks per tile); on GEMM1 it measured slower.
#include "gemm_fp8.cuh"
#include "gemm_sched.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBK8 = 128;        // e4m3 elements per 128-byte swizzle row = one scale block
constexpr int kUK8 = 32;         // K per tcgen05.mma kind::f8f6f4
constexpr int kBN8 = 256;
template <Fp8Epi EPI>
struct F8Cfg {
  static constexpr int kEpiWarps = EPI == Fp8Epi::kSwiGLU ? 8 : 16;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
};
constexpr int kABytes8 = kBM * 128;
constexpr int kBBytes8 = kBN8 * 128;
constexpr int kStage8 = kABytes8 + kBBytes8;
constexpr int kStages8 = 4;
constexpr int kAux8 = 12288;
constexpr int kSmem8 = 1024 + kStages8 * kStage8 + kAux8;

__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, 256;" ::: "memory");  // the 8 epilogue warps (SwiGLU)
}

__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  return (uint32_t)f32_to_e4m3(a) | ((uint32_t)f32_to_e4m3(b) << 8) | ((uint32_t)f32_to_e4m3(c) << 16) |
         ((uint32_t)f32_to_e4m3(d) << 24);
}

template <Fp8Epi EPI>
__global__ void __launch_bounds__(F8Cfg<EPI>::kThreads, 1)
    tc_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                       const Fp8GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages8 * kABytes8;
  uint8_t* aux = smem + kStages8 * kStage8;
  uint64_t* full = reinterpret_cast<uint64_t*>(aux);
  uint64_t* empty = full + kStages8;
  uint64_t* tfull = empty + kStages8;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* s_tp = reinterpret_cast<int*>(aux + 256);
  int* s_mt = s_tp + (kMaxGroups + 1);
  int* s_off = s_mt + kMaxGroups;
  float* s_amax = reinterpret_cast<float*>(s_off + kMaxGroups + 1);  // [2][128]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == 0) {
    const int G0 = p.groups0;
    const int per = (G0 + 31) / 32;
    const int beg = min(lane * per, G0), end = min(beg + per, G0);
    int sum = 0;
    for (int g = beg; g < end; ++g) {
      const int o0 = p.offsets0[g], o1 = p.offsets0[g + 1];
      s_off[g] = o0;
      const int mt = (o1 - o0 + kBM - 1) / kBM;
      s_mt[g] = mt;
      sum += mt;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int g = beg; g < end; ++g) {
      s_tp[g] = run * p.n_tiles0;
      run += s_mt[g];
    }
    if (lane == 31) {
      s_tp[G0] = incl * p.n_tiles0;
      if (G0 > 0) s_off[G0] = p.offsets0[G0];
    }
  }
  __syncthreads();

  Sched sch;
  sch.tp = s_tp;
  sch.mt = s_mt;
  sch.off = s_off;
  sch.groups0 = p.groups0;
  sch.tiles0 = s_tp[p.groups0];
  sch.n_tiles0 = p.n_tiles0;
  sch.n_tiles1 = p.n_tiles1;
  sch.rows1 = p.rows1;
  sch.mt1 = (p.rows1 + kBM - 1) / kBM;
  sch.total = sch.tiles0 + sch.mt1 * p.n_tiles1;
  if ((int)blockIdx.x >= sch.total) return;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kStages8; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], F8Cfg<EPI>::kEpiWarps);
    }
    ptx::mbar_init(mma_done, 1);
    ptx::fence_barrier_init();
    if (p.groups0 > 0) {
      ptx::prefetch_tmap(&tmA0);
      ptx::prefetch_tmap(&tmB0);
    }
    if (p.rows1 > 0) {
      ptx::prefetch_tmap(&tmA1);
      ptx::prefetch_tmap(&tmB1);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ================= TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < sch.total && ok; L += gridDim.x) {
        const Tile t = sch.decode(L);
        const int kbs = t.seg ? p.k_blocks1 : p.k_blocks0;
        const CUtensorMap* ma = t.seg ? &tmA1 : &tmA0;
        const CUtensorMap* mb = t.seg ? &tmB1 : &tmB0;
        for (int kb = 0; kb < kbs; ++kb) {
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1, p.err)) {
            set_error(p.err, kDevTimeoutProducer);
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[stage], kStage8);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          uint8_t* a_dst = sA + stage * kABytes8;
          uint8_t* b_dst = sB + stage * kBBytes8;
          const int k0 = kb * kBK8;
          ptx::tma_load_2d(a_dst, ma, &full[stage], k0, t.row0);
          if constexpr (EPI == Fp8Epi::kSwiGLU) {
            int e, nrow;
            if (t.seg == 0) {
              e = t.group;
              nrow = t.n * 128;
            } else {
              const int per = p.I / 128;
              e = t.n / per;
              nrow = (t.n % per) * 128;
            }
            ptx::tma_load_3d(b_dst + 0 * 8192, mb, &full[stage], k0, nrow, e);
            ptx::tma_load_3d(b_dst + 1 * 8192, mb, &full[stage], k0, p.I + nrow, e);
            ptx::tma_load_3d(b_dst + 2 * 8192, mb, &full[stage], k0, nrow + 64, e);
            ptx::tma_load_3d(b_dst + 3 * 8192, mb, &full[stage], k0, p.I + nrow + 64, e);
          } else {
            if (t.seg == 0) {
              ptx::tma_load_3d(b_dst, mb, &full[stage], k0, t.n * kBN8, t.group);
            } else {
              ptx::tma_load_3d(b_dst, mb, &full[stage], k0 % p.I, t.n * kBN8, k0 / p.I);
            }
          }
          if (++stage == kStages8) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      for (int s = 0; s < kStages8; ++s) {
        if (armed & (1u << s)) {
          if (!ptx::mbar_wait(&full[s], (armed_parity >> s) & 1u, nullptr)) set_error(p.err, kDevTimeoutDrain);
        }
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer: one fresh accumulation per K block
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_e4m3(kBM, kBN8);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t g = 0;  // K blocks issued so far (selects the TMEM buffer)
      bool ok = true;
      for (int L = blockIdx.x; L < sch.total && ok; L += gridDim.x) {
        const Tile t = sch.decode(L);
        const int kbs = t.seg ? p.k_blocks1 : p.k_blocks0;
        for (int kb = 0; kb < kbs; ++kb, ++g) {
          const uint32_t b = g & 1;
          if (!ptx::mbar_wait(&tempty[b], ((g >> 1) & 1) ^ 1, p.err) ||
              !ptx::mbar_wait(&full[stage], phase, p.err)) {
            set_error(p.err, kDevTimeoutMma);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem_base + b * kBN8;
          const uint64_t adesc = ptx::smem_desc_sw128(ptx::smem_u32(sA + stage * kABytes8));
          const uint64_t bdesc = ptx::smem_desc_sw128(ptx::smem_u32(sB + stage * kBBytes8));
#pragma unroll
          for (int k = 0; k < kBK8 / kUK8; ++k) ptx::mma_f8(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, k != 0);
          ptx::tc_commit(&empty[stage]);
          ptx::tc_commit(&tfull[b]);
          if (++stage == kStages8) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      ptx::tc_commit(mma_done);
      if (!ptx::mbar_wait(mma_done, 0, nullptr)) set_error(p.err, kDevTimeoutDrain);
    }
  } else {
    if constexpr (EPI == Fp8Epi::kSwiGLU) {
      // ================= epilogue (warps 2..9)
      const int q = warp & 3;
      const int half = (warp - 2) >> 2;
      const int r_in_tile = 32 * q + lane;
      uint32_t g = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < sch.total; L += gridDim.x) {
        const Tile t = sch.decode(L);
        const int kbs = t.seg ? p.k_blocks1 : p.k_blocks0;
        const int row = t.row0 + r_in_tile;
        const int rows_total = t.seg ? p.rows1 : p.rows_total0;
        const bool valid = row < t.row_end;
        const float* sa_base = t.seg ? p.a_scale1 : p.a_scale0;
        // per-tile weight-scale addressing
        const float* sb_base;
        int sb_stride_kb = 1;
        int rb0 = 0, rb1 = 0;  // scale rows (128-row weight blocks) for this half's two 64-col parts
        if constexpr (EPI == Fp8Epi::kSwiGLU) {
          const int nblk = p.I / 128;  // 128-row blocks per projection
          int e, nn;
          if (t.seg == 0) {
            e = t.group;
            nn = t.n;
          } else {
            e = t.n / nblk;
            nn = t.n % nblk;
          }
          const int kbk = t.seg ? p.k_blocks1 : p.k_blocks0;  // d / 128
          sb_base = (t.seg ? p.b_scale1 : p.b_scale0) + (size_t)e * (2 * nblk) * kbk;
          rb0 = nn;          // gate block
          rb1 = nblk + nn;   // up block
          sb_stride_kb = kbk;
        } else {
          const int nbd = p.N / 128;  // d / 128 row blocks of W2
          const int kpe = p.I / 128;  // K blocks per expert
          sb_base = t.seg ? p.b_scale1 : p.b_scale0 + (size_t)t.group * nbd * kpe;
          rb0 = rb1 = t.n * 2 + half;
          sb_stride_kb = kpe;
        }
        float acc[128];
  #pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
        for (int kb = 0; kb < kbs; ++kb, ++g) {
          const uint32_t b = g & 1;
          if (ok && !ptx::mbar_wait(&tfull[b], (g >> 1) & 1, p.err)) {
            set_error(p.err, kDevTimeoutEpilogue);
            ok = false;
          }
          ptx::tc_fence_after();
          const float sa = (row < rows_total && ok) ? __ldg(sa_base + (size_t)kb * rows_total + row) : 0.0f;
          float f0, f1;
          if constexpr (EPI == Fp8Epi::kSwiGLU) {
            f0 = sa * __ldg(sb_base + (size_t)rb0 * sb_stride_kb + kb);
            f1 = sa * __ldg(sb_base + (size_t)rb1 * sb_stride_kb + kb);
          } else {
            // shared segment: K runs over S experts of I columns each
            const int e = t.seg ? (kb * 128) / p.I : 0;
            const int kk = t.seg ? ((kb * 128) % p.I) / 128 : kb;
            const float* sb = t.seg ? p.b_scale1 + (size_t)e * (p.N / 128) * (p.I / 128) : sb_base;
            f0 = f1 = sa * __ldg(sb + (size_t)rb0 * sb_stride_kb + kk);
          }
          if (ok) {
            const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16) + b * kBN8 + half * 128;
  #pragma unroll
            for (int c = 0; c < 4; ++c) {
              float v[32];
              ptx::tmem_ld32(tb + c * 32, v);
              const float f = (c < 2) ? f0 : f1;
  #pragma unroll
              for (int j = 0; j < 32; ++j) acc[c * 32 + j] = fmaf(v[j], f, acc[c * 32 + j]);
            }
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&tempty[b]);
        }
        if constexpr (EPI == Fp8Epi::kSwiGLU) {
          // h = silu(gate) * up for this half's 64 intermediate columns, then the
          // 1x128 e4m3 tile shared with the other half of the row
          float amax = 0.0f;
  #pragma unroll
          for (int j = 0; j < 64; ++j) {
            acc[j] = silu(acc[j]) * acc[64 + j];
            amax = fmaxf(amax, fabsf(acc[j]));
          }
          s_amax[half * 128 + r_in_tile] = amax;
          epi_bar();
          amax = fmaxf(amax, s_amax[(half ^ 1) * 128 + r_in_tile]);
          epi_bar();  // s_amax is rewritten by the next tile
          const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
          if (valid) {
            uint8_t* out = static_cast<uint8_t*>(t.seg ? p.out1 : p.out0);
            const int ldo = t.seg ? p.ldo1 : p.ldo0;
            uint4* dst = reinterpret_cast<uint4*>(out + (size_t)row * ldo + t.n * 128 + half * 64);
  #pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 w;
              w.x = pack4_e4m3(__fdiv_rn(acc[16 * v + 0], scale), __fdiv_rn(acc[16 * v + 1], scale),
                               __fdiv_rn(acc[16 * v + 2], scale), __fdiv_rn(acc[16 * v + 3], scale));
              w.y = pack4_e4m3(__fdiv_rn(acc[16 * v + 4], scale), __fdiv_rn(acc[16 * v + 5], scale),
                               __fdiv_rn(acc[16 * v + 6], scale), __fdiv_rn(acc[16 * v + 7], scale));
              w.z = pack4_e4m3(__fdiv_rn(acc[16 * v + 8], scale), __fdiv_rn(acc[16 * v + 9], scale),
                               __fdiv_rn(acc[16 * v + 10], scale), __fdiv_rn(acc[16 * v + 11], scale));
              w.w = pack4_e4m3(__fdiv_rn(acc[16 * v + 12], scale), __fdiv_rn(acc[16 * v + 13], scale),
                               __fdiv_rn(acc[16 * v + 14], scale), __fdiv_rn(acc[16 * v + 15], scale));
              dst[v] = w;
            }
            if (half == 0) {
              float* hs = t.seg ? p.out_scale1 : p.out_scale0;
              hs[(size_t)t.n * rows_total + row] = scale;
            }
          }
        } else {
          if (valid) {
            __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(t.seg ? p.out1 : p.out0);
            const int ldo = t.seg ? p.ldo1 : p.ldo0;
            const size_t o = (size_t)row * ldo + t.n * kBN8 + half * 128;
  #pragma unroll
            for (int c = 0; c < 4; ++c) {
              if constexpr (EPI == Fp8Epi::kCombine) add_bf16x32(acc + 32 * c, p.radd + o + 32 * c, 1.0f);
              store_bf16x32(out + o + 32 * c, acc + 32 * c);
            }
          }
        }
      }
    } else {
      // ================= epilogue (warps 2..17)
      const int q = warp & 3;
      const int slice = (warp - 2) >> 2;  // 0..3
      const int r_in_tile = 32 * q + lane;
      // SwiGLU: this warp's 32 h columns are 32 slice .. 32 slice + 31 of the
      // tile's 128; their gate accumulators start at column ga (B tile rows are
      // [gate 0..63 | up 0..63 | gate 64..127 | up 64..127]), the up ones at ga + 64
      const int ga = slice < 2 ? 32 * slice : 128 + 32 * (slice - 2);
      uint32_t g = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < sch.total; L += gridDim.x) {
        const Tile t = sch.decode(L);
        const int kbs = t.seg ? p.k_blocks1 : p.k_blocks0;
        const int row = t.row0 + r_in_tile;
        const int rows_total = t.seg ? p.rows1 : p.rows_total0;
        const bool valid = row < t.row_end;
        const float* sa_base = t.seg ? p.a_scale1 : p.a_scale0;
        // per-tile weight-scale addressing
        const float* sb_base;
        int sb_stride_kb = 1;
        int rb0 = 0, rb1 = 0;  // scale rows (128-row weight blocks) of this warp's two 32-column parts
        if constexpr (EPI == Fp8Epi::kSwiGLU) {
          const int nblk = p.I / 128;  // 128-row blocks per projection
          int e, nn;
          if (t.seg == 0) {
            e = t.group;
            nn = t.n;
          } else {
            e = t.n / nblk;
            nn = t.n % nblk;
          }
          const int kbk = t.seg ? p.k_blocks1 : p.k_blocks0;  // d / 128
          sb_base = (t.seg ? p.b_scale1 : p.b_scale0) + (size_t)e * (2 * nblk) * kbk;
          rb0 = nn;          // gate block
          rb1 = nblk + nn;   // up block
          sb_stride_kb = kbk;
        } else {
          const int nbd = p.N / 128;  // d / 128 row blocks of W2
          const int kpe = p.I / 128;  // K blocks per expert
          sb_base = t.seg ? p.b_scale1 : p.b_scale0 + (size_t)t.group * nbd * kpe;
          rb0 = rb1 = t.n * 2 + (slice >> 1);  // columns 64 slice .. 64 slice + 63
          sb_stride_kb = kpe;
        }
        float acc[64];
  #pragma unroll
        for (int j = 0; j < 64; ++j) acc[j] = 0.0f;
        for (int kb = 0; kb < kbs; ++kb, ++g) {
          const uint32_t b = g & 1;
          if (ok && !ptx::mbar_wait(&tfull[b], (g >> 1) & 1, p.err)) {
            set_error(p.err, kDevTimeoutEpilogue);
            ok = false;
          }
          ptx::tc_fence_after();
          const float sa = (row < rows_total && ok) ? __ldg(sa_base + (size_t)kb * rows_total + row) : 0.0f;
          float f0, f1;
          if constexpr (EPI == Fp8Epi::kSwiGLU) {
            f0 = sa * __ldg(sb_base + (size_t)rb0 * sb_stride_kb + kb);
            f1 = sa * __ldg(sb_base + (size_t)rb1 * sb_stride_kb + kb);
          } else {
            // shared segment: K runs over S experts of I columns each
            const int e = t.seg ? (kb * 128) / p.I : 0;
            const int kk = t.seg ? ((kb * 128) % p.I) / 128 : kb;
            const float* sb = t.seg ? p.b_scale1 + (size_t)e * (p.N / 128) * (p.I / 128) : sb_base;
            f0 = f1 = sa * __ldg(sb + (size_t)rb0 * sb_stride_kb + kk);
          }
          if (ok) {
            const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16) + b * kBN8;
            const uint32_t c0 = EPI == Fp8Epi::kSwiGLU ? ga : 64 * slice;
            const uint32_t c1 = EPI == Fp8Epi::kSwiGLU ? ga + 64 : 64 * slice + 32;
            // 16 columns per load keeps the temporaries within the 96
            // registers a thread of a 576-thread block has
  #pragma unroll
            for (int h = 0; h < 4; ++h) {
              float v[16];
              ptx::tmem_ld16(tb + (h < 2 ? c0 : c1) + 16 * (h & 1), v);
              const float f = h < 2 ? f0 : f1;
  #pragma unroll
              for (int j = 0; j < 16; ++j) acc[16 * h + j] = fmaf(v[j], f, acc[16 * h + j]);
            }
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&tempty[b]);
        }
        if constexpr (EPI == Fp8Epi::kSwiGLU) {
          // h = silu(gate) * up for this warp's 32 intermediate columns, then
          // the 1x128 e4m3 tile shared with the three other slices of the row
          float amax = 0.0f;
  #pragma unroll
          for (int j = 0; j < 32; ++j) {
            acc[j] = silu(acc[j]) * acc[32 + j];
            amax = fmaxf(amax, fabsf(acc[j]));
          }
          s_amax[slice * 128 + r_in_tile] = amax;
          epi_bar();
  #pragma unroll
          for (int o = 0; o < 4; ++o) amax = fmaxf(amax, s_amax[o * 128 + r_in_tile]);
          epi_bar();  // s_amax is rewritten by the next tile
          const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
          if (valid) {
            uint8_t* out = static_cast<uint8_t*>(t.seg ? p.out1 : p.out0);
            const int ldo = t.seg ? p.ldo1 : p.ldo0;
            uint4* dst = reinterpret_cast<uint4*>(out + (size_t)row * ldo + t.n * 128 + slice * 32);
  #pragma unroll
            for (int v = 0; v < 2; ++v) {
              uint4 w;
              w.x = pack4_e4m3(__fdiv_rn(acc[16 * v + 0], scale), __fdiv_rn(acc[16 * v + 1], scale),
                               __fdiv_rn(acc[16 * v + 2], scale), __fdiv_rn(acc[16 * v + 3], scale));
              w.y = pack4_e4m3(__fdiv_rn(acc[16 * v + 4], scale), __fdiv_rn(acc[16 * v + 5], scale),
                               __fdiv_rn(acc[16 * v + 6], scale), __fdiv_rn(acc[16 * v + 7], scale));
              w.z = pack4_e4m3(__fdiv_rn(acc[16 * v + 8], scale), __fdiv_rn(acc[16 * v + 9], scale),
                               __fdiv_rn(acc[16 * v + 10], scale), __fdiv_rn(acc[16 * v + 11], scale));
              w.w = pack4_e4m3(__fdiv_rn(acc[16 * v + 12], scale), __fdiv_rn(acc[16 * v + 13], scale),
                               __fdiv_rn(acc[16 * v + 14], scale), __fdiv_rn(acc[16 * v + 15], scale));
              dst[v] = w;
            }
            if (slice == 0) {
              float* hs = t.seg ? p.out_scale1 : p.out_scale0;
              hs[(size_t)t.n * rows_total + row] = scale;
            }
          }
        } else {
          if (valid) {
            __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(t.seg ? p.out1 : p.out0);
            const int ldo = t.seg ? p.ldo1 : p.ldo0;
            const size_t o = (size_t)row * ldo + t.n * kBN8 + slice * 64;
  #pragma unroll
            for (int c = 0; c < 2; ++c) {
              if constexpr (EPI == Fp8Epi::kCombine) add_bf16x32(acc + 32 * c, p.radd + o + 32 * c, 1.0f);
              store_bf16x32(out + o + 32 * c, acc + 32 * c);
            }
          }
        }
      }
    }
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

template <Fp8Epi EPI>
cudaError_t launch_fp8_one(const Fp8GemmLaunch& L) {
  auto kern = tc_gemm_fp8_kernel<EPI>;
  static int attr_done[64] = {};
  cudaError_t e = set_smem_once(kern, kSmem8, attr_done);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, F8Cfg<EPI>::kThreads, kSmem8, L.stream>>>(L.a0, L.b0, L.a1, L.b1, L.p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8_gemm(const Fp8GemmLaunch& L) {
  if (L.p.groups0 > kMaxGroups) return cudaErrorInvalidValue;
  switch (L.epi) {
    case Fp8Epi::kSwiGLU: return launch_fp8_one<Fp8Epi::kSwiGLU>(L);
    case Fp8Epi::kStore: return launch_fp8_one<Fp8Epi::kStore>(L);
    case Fp8Epi::kCombine: return launch_fp8_one<Fp8Epi::kCombine>(L);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
