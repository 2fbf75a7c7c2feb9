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
// Roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer, warps 2 and
// 3 idle, warps 4..11 epilogue; epilogue warp w drains TMEM lane quarter
// w % 4 and column half (w - 4) / 4 (128 of the tile's 256 columns) into 128
// fp32 accumulators. setmaxnreg gives the epilogue warpgroups 232 registers a
// thread (the control warpgroup keeps 40), so two 32-column TMEM loads stay
// in flight without spilling; each K block's scales are loaded while the
// block before it drains, and the accumulator buffer is released before the
// last FMAs of the block. GEMM1 quantises h to e4m3 in its epilogue; the
// down projections write bf16 rows through a staging block per warp.
#include "gemm_fp8.cuh"
#include "gemm_sched.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBK8 = 128;        // e4m3 elements per 128-byte swizzle row = one scale block
constexpr int kUK8 = 32;         // K per tcgen05.mma kind::f8f6f4
constexpr int kBN8 = 256;
// Three warpgroups; setmaxnreg moves registers from the control warpgroup
// (producer, MMA issuer, two idle warps) to the two epilogue warpgroups, so
// that 128 accumulators and two 32-column TMEM loads in flight fit without
// spilling.
struct F8Cfg {
  static constexpr int kCtlWarps = 4;
  static constexpr int kEpiWarps = 8;
  static constexpr int kThreads = 32 * (kCtlWarps + kEpiWarps);
  static constexpr int kLaunchRegs = 168;  // 3 warps per SM sub-partition: 3 x 32 x 168 <= 16384
  static constexpr int kCtlRegs = 40;
  static constexpr int kEpiRegs = 232;
};
static_assert(F8Cfg::kThreads * F8Cfg::kLaunchRegs ==
                  32 * F8Cfg::kCtlWarps * F8Cfg::kCtlRegs + 32 * F8Cfg::kEpiWarps * F8Cfg::kEpiRegs,
              "the register split must hand out exactly the registers the block is launched with");
constexpr int kABytes8 = kBM * 128;
constexpr int kBBytes8 = kBN8 * 128;
constexpr int kStage8 = kABytes8 + kBBytes8;
constexpr int kStages8 = 4;
constexpr int kAux8 = 12288;
constexpr int kStg8 = F8Cfg::kEpiWarps * kRowStageBytes;  // bf16 output staging, one block per epilogue warp
constexpr int kSmem8 = 1024 + kStages8 * kStage8 + kAux8 + kStg8;

__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, 256;" ::: "memory");  // the 8 epilogue warps (SwiGLU)
}



__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  return (uint32_t)f32_to_e4m3(a) | ((uint32_t)f32_to_e4m3(b) << 8) | ((uint32_t)f32_to_e4m3(c) << 16) |
         ((uint32_t)f32_to_e4m3(d) << 24);
}

template <Fp8Epi EPI>
__global__ void __launch_bounds__(F8Cfg::kThreads, 1)
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
  uint8_t* s_stage = aux + kAux8;

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
      ptx::mbar_init(&tempty[a], F8Cfg::kEpiWarps);
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

  if (warp < F8Cfg::kCtlWarps) {
    // the register split is issued by whole warpgroups, ahead of each role's code
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(F8Cfg::kCtlRegs));
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
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(F8Cfg::kEpiRegs));
    // ================= epilogue (warps 4..11)
    const int q = warp & 3;
    const int half = (warp - F8Cfg::kCtlWarps) >> 2;  // columns 128 half .. 128 half + 127 of the tile
    const int r_in_tile = 32 * q + lane;
    uint8_t* stg = s_stage + (warp - F8Cfg::kCtlWarps) * kRowStageBytes;
    uint32_t g = 0;
    bool ok = true;
    for (int L = blockIdx.x; L < sch.total; L += gridDim.x) {
      const Tile t = sch.decode(L);
      const int kbs = t.seg ? p.k_blocks1 : p.k_blocks0;
      const int row = t.row0 + r_in_tile;
      const int rows_total = t.seg ? p.rows1 : p.rows_total0;
      const bool valid = row < t.row_end;
      const float* sa_base = t.seg ? p.a_scale1 : p.a_scale0;
      // weight scales of this warp's columns: sb0p for the first 64, sb1p for
      // the last 64, at offset kb (SwiGLU) or the block's place in [S, N/128, I/128]
      const float* sb0p;
      const float* sb1p;
      int nbd = 0, kpe = 1;
      if constexpr (EPI == Fp8Epi::kSwiGLU) {
        // B tile rows [gate 0..63 | up 0..63 | gate 64..127 | up 64..127]:
        // this half holds gate and up of h columns 64 half .. 64 half + 63
        const int nblk = p.I / 128;  // 128-row blocks per projection
        const int e = t.seg ? t.n / nblk : t.group;
        const int nn = t.seg ? t.n % nblk : t.n;
        const float* sb_base = (t.seg ? p.b_scale1 : p.b_scale0) + (size_t)e * (2 * nblk) * kbs;
        sb0p = sb_base + (size_t)nn * kbs;           // gate block
        sb1p = sb_base + (size_t)(nblk + nn) * kbs;  // up block
      } else {
        // down projection: K runs over S experts of I columns each in the
        // shared segment, over one expert's I in the routed one
        nbd = p.N / 128;
        kpe = p.I / 128;
        const float* sb_base = t.seg ? p.b_scale1 : p.b_scale0 + (size_t)t.group * nbd * kpe;
        sb0p = sb1p = sb_base + (size_t)(t.n * 2 + half) * kpe;
      }
      // offset of the next block's weight scale: kb (SwiGLU); in the down
      // projections the K block within an expert, plus nbd * kpe per expert
      // passed (stepped, not divided, per block)
      int sb_k = 0, sb_e = 0;
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
      // the scales of block kb + 1 are loaded while block kb drains
      const bool row_in = row < rows_total;
      float sa_n = 0.0f, sb0_n = 0.0f, sb1_n = 0.0f;
      if (kbs > 0) {
        sa_n = row_in ? __ldg(sa_base + row) : 0.0f;
        sb0_n = __ldg(sb0p);
        sb1_n = EPI == Fp8Epi::kSwiGLU ? __ldg(sb1p) : sb0_n;
      }
      for (int kb = 0; kb < kbs; ++kb, ++g) {
        const uint32_t b = g & 1;
        const float f0 = sa_n * sb0_n, f1 = sa_n * sb1_n;
        if (kb + 1 < kbs) {
          int o;
          if constexpr (EPI == Fp8Epi::kSwiGLU) {
            o = kb + 1;
          } else {
            if (++sb_k == kpe) {
              sb_k = 0;
              sb_e += nbd * kpe;
            }
            o = sb_e + sb_k;
          }
          sa_n = row_in ? __ldg(sa_base + (size_t)(kb + 1) * rows_total + row) : 0.0f;
          sb0_n = __ldg(sb0p + o);
          sb1_n = EPI == Fp8Epi::kSwiGLU ? __ldg(sb1p + o) : sb0_n;
        }
        if (ok && !ptx::mbar_wait(&tfull[b], (g >> 1) & 1, p.err)) {
          set_error(p.err, kDevTimeoutEpilogue);
          ok = false;
        }
        ptx::tc_fence_after();
        float v0[32], v1[32];
        const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16) + b * kBN8 + half * 128;
        if (ok) {
          // columns 0..63 of this half, two loads in flight
          ptx::tmem_ld32_nowait(tb, v0);
          ptx::tmem_ld32_nowait(tb + 32, v1);
          ptx::tmem_wait_ld(v0);
          ptx::tmem_wait_ld(v1);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            ptx::ffma2(acc[j], acc[j + 1], v0[j], v0[j + 1], f0);
            ptx::ffma2(acc[32 + j], acc[33 + j], v1[j], v1[j + 1], f0);
          }
          // columns 64..127; the buffer is released before their FMAs
          ptx::tmem_ld32_nowait(tb + 64, v0);
          ptx::tmem_ld32_nowait(tb + 96, v1);
          ptx::tmem_wait_ld(v0);
          ptx::tmem_wait_ld(v1);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&tempty[b]);
        if (ok) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            ptx::ffma2(acc[64 + j], acc[65 + j], v0[j], v0[j + 1], f1);
            ptx::ffma2(acc[96 + j], acc[97 + j], v1[j], v1[j + 1], f1);
          }
        }
      }
      if constexpr (EPI == Fp8Epi::kSwiGLU) {
        // h = silu(gate) * up for this half's 64 intermediate columns, then the
        // 1x128 e4m3 tile shared with the other half of the row
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          acc[j] = silu_fast(acc[j]) * acc[64 + j];
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
        // bf16 rows through the warp's staging block, 32 columns at a time
        // (kCombine adds the routed sum of the row first)
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(t.seg ? p.out1 : p.out0);
        const int ldo = t.seg ? p.ldo1 : p.ldo0;
        const int rbase = t.row0 + 32 * q;
        const int nrows = max(0, min(32, t.row_end - rbase));
        const size_t col = (size_t)t.n * kBN8 + half * 128;
        uint8_t* base = reinterpret_cast<uint8_t*>(out + (size_t)rbase * ldo + col);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if constexpr (EPI == Fp8Epi::kCombine) {
            if (valid) add_bf16x32(acc + 32 * c, p.radd + (size_t)row * ldo + col + 32 * c, 1.0f);
          }
          uint4 w[4];
          pack_bf16x32(acc + 32 * c, w);
          warp_store_rows64(stg, lane, w, base + c * 64, (size_t)ldo * 2, nrows);
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
  {
    // setmaxnreg.inc waits until the registers it asks for are free: refuse
    // to launch unless the block starts with exactly the registers it splits
    static int regs_ok = 0;
    if (!regs_ok) {
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != F8Cfg::kLaunchRegs) return cudaErrorInvalidConfiguration;
      regs_ok = 1;
    }
  }
  kern<<<L.grid, F8Cfg::kThreads, kSmem8, L.stream>>>(L.a0, L.b0, L.a1, L.b1, L.p);
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
