// FP8 (e4m3) persistent grouped GEMM with the tensor core's own block
// scaling: tcgen05.mma kind::mxf8f6f4.block_scale, one UE8M0 (power-of-two)
// scale per 32 K values of every A and B row, accumulated over the whole K in
// TMEM. It serves the FP8 path when its tiles carry power-of-two scales
// ("DeepSeek-V3技术报告" digest, mpbf.cn, section 3.1: FP8 GEMM inputs with
// per-tile scale factors and fp32 accumulation; the power-of-two scale rule is
// this library's option). With such scales the product of a K block scaled by
// scale_a * scale_b is exact, so scaling inside the MMA gives the same sums
// as scaling the per-block partial products, and no promotion pass is needed.
//
// Operands as in the fp32-scale kernel: A rows in 1x128 e4m3 tiles with one
// scale per (row, tile), tile-major [K/128, rows]; B (weights) in 128x128
// e4m3 blocks with one scale per block. Each 128-wide K block is one pipeline
// stage and four MMAs of K = 32 that share its scales.
//
// Roles (352 threads): warp 0 TMA producer; warp 1 MMA issuer and TMEM owner;
// warp 2 scale producer: it turns each stage's fp32 power-of-two scales into
// UE8M0 bytes in shared memory, laid out for tcgen05.cp; warps 3..10
// epilogue (warp w drains TMEM lane quarter w % 4, column half (w - 3) / 4).
//
// TMEM: columns 0..255 hold the 128 x 256 fp32 accumulator (one buffer: the
// epilogue copies it to registers and releases it before its own math);
// columns 256..319 hold four scale slots of 16 columns, one per pipeline
// stage (A scales in columns 0..3 of the slot, B scales in 4..11). A
// tcgen05.cp of 32 rows x 16 bytes repeated over the four lane quarters
// fills both layouts the MMA reads from one 512-byte block per 128 rows in
// which word 4l + c holds the scale of row 32c + l.
#include "gemm_fp8.cuh"
#include "gemm_sched.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBKx = 128;  // e4m3 elements per 128-byte swizzle row = one scale block
constexpr int kUKx = 32;   // K per tcgen05.mma kind::mxf8f6f4
constexpr int kBNx = 256;
constexpr int kThreadsX = 352;
constexpr int kStagesX = 4;
constexpr int kABytesX = kBM * 128;
constexpr int kBBytesX = kBNx * 128;
constexpr int kStageX = kABytesX + kBBytesX;
constexpr int kSfaBytes = 512;   // 128 A rows, one word each (4 copies of the byte)
constexpr int kSfbBytes = 1024;  // 256 B rows
constexpr int kSfBytes = kSfaBytes + kSfbBytes;
constexpr int kAuxX = 8192;
constexpr int kStgWarp = kRowStageBytes;  // per epilogue warp: 32 rows x 64 bytes of output
constexpr int kSmemX = 1024 + kStagesX * (kStageX + kSfBytes) + kAuxX + 8 * kStgWarp;
constexpr uint32_t kSfCol = 256;  // first TMEM column of the scale slots
constexpr uint32_t kSfSlot = 16;  // TMEM columns per slot

__device__ __forceinline__ void epi_bar_x() {
  asm volatile("bar.sync 1, 256;" ::: "memory");  // the 8 epilogue warps
}

__device__ __forceinline__ uint32_t pack4_e4m3_x(float a, float b, float c, float d) {
  return (uint32_t)f32_to_e4m3(a) | ((uint32_t)f32_to_e4m3(b) << 8) | ((uint32_t)f32_to_e4m3(c) << 16) |
         ((uint32_t)f32_to_e4m3(d) << 24);
}

// Position in this CTA's sequence of (tile, K block) stages.
struct Cursor {
  int L, kb, kbs;
  Tile t;
};

__device__ __forceinline__ void cursor_load_tile(Cursor& c, const Sched& sch, const Fp8GemmParams& p) {
  if (c.L < sch.total) {
    c.t = sch.decode(c.L);
    c.kbs = c.t.seg ? p.k_blocks1 : p.k_blocks0;
  }
}

__device__ __forceinline__ void cursor_next(Cursor& c, const Sched& sch, const Fp8GemmParams& p) {
  if (++c.kb == c.kbs) {
    c.kb = 0;
    c.L += gridDim.x;
    cursor_load_tile(c, sch, p);
  }
}

// The scales of one stage as this lane needs them: a[c] = A scale of tile row
// 32c + lane (1 past the matrix end); b[0], b[1] = the two weight-block
// scales of the tile's B rows (SwiGLU: gate block, up block; otherwise the
// blocks of B rows 0..127 and 128..255).
template <Fp8Epi EPI>
__device__ __forceinline__ void load_stage_scales(const Fp8GemmParams& p, const Tile& t, int kb, int lane,
                                                  float (&a)[4], float (&b)[2]) {
  const float* sa = t.seg ? p.a_scale1 : p.a_scale0;
  const int rows_total = t.seg ? p.rows1 : p.rows_total0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int row = t.row0 + 32 * c + lane;
    a[c] = row < rows_total ? __ldg(sa + (size_t)kb * rows_total + row) : 1.0f;
  }
  if constexpr (EPI == Fp8Epi::kSwiGLU) {
    const int nblk = p.I / 128;
    const int e = t.seg ? t.n / nblk : t.group;
    const int nn = t.seg ? t.n % nblk : t.n;
    const int kbk = t.seg ? p.k_blocks1 : p.k_blocks0;  // d / 128
    const float* sb = (t.seg ? p.b_scale1 : p.b_scale0) + (size_t)e * (2 * nblk) * kbk;
    b[0] = __ldg(sb + (size_t)nn * kbk + kb);
    b[1] = __ldg(sb + (size_t)(nblk + nn) * kbk + kb);
  } else {
    const int nbd = p.N / 128;  // 128-row blocks of W2 (d / 128)
    const int kpe = p.I / 128;  // K blocks per expert
    const float* sb;
    int kk;
    if (t.seg == 0) {
      sb = p.b_scale0 + (size_t)t.group * nbd * kpe;
      kk = kb;
    } else {
      // shared segment: K runs over the S experts, I columns each
      sb = p.b_scale1 + (size_t)((kb * 128) / p.I) * nbd * kpe;
      kk = ((kb * 128) % p.I) / 128;
    }
    b[0] = __ldg(sb + (size_t)(2 * t.n) * kpe + kk);
    b[1] = __ldg(sb + (size_t)(2 * t.n + 1) * kpe + kk);
  }
}

template <Fp8Epi EPI>
__global__ void __launch_bounds__(kThreadsX, 1)
    tc_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                      const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                      const Fp8GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStagesX * kABytesX;
  uint8_t* sSF = smem + kStagesX * kStageX;  // [stage][SFA 512 | SFB 1024]
  uint8_t* aux = sSF + kStagesX * kSfBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(aux);  // TMA bytes landed
  uint64_t* sfull = full + kStagesX;                  // scale bytes written
  uint64_t* empty = sfull + kStagesX;
  uint64_t* tfull = empty + kStagesX;
  uint64_t* tempty = tfull + 1;
  uint64_t* mma_done = tempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* s_tp = reinterpret_cast<int*>(aux + 256);
  int* s_mt = s_tp + (kMaxGroups + 1);
  int* s_off = s_mt + kMaxGroups;
  float* s_amax = reinterpret_cast<float*>(s_off + kMaxGroups + 1);  // [2][128]
  uint8_t* s_stage_out = aux + kAuxX;                                 // [8 warps][2048]

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
    for (int s = 0; s < kStagesX; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&sfull[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(tfull, 1);
    ptx::mbar_init(tempty, 8);
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
          ptx::mbar_arrive_expect_tx(&full[stage], kStageX);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          uint8_t* a_dst = sA + stage * kABytesX;
          uint8_t* b_dst = sB + stage * kBBytesX;
          const int k0 = kb * kBKx;
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
              ptx::tma_load_3d(b_dst, mb, &full[stage], k0, t.n * kBNx, t.group);
            } else {
              ptx::tma_load_3d(b_dst, mb, &full[stage], k0 % p.I, t.n * kBNx, k0 / p.I);
            }
          }
          if (++stage == kStagesX) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      for (int s = 0; s < kStagesX; ++s) {
        if (armed & (1u << s)) {
          if (!ptx::mbar_wait(&full[s], (armed_parity >> s) & 1u, nullptr)) set_error(p.err, kDevTimeoutDrain);
        }
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_mx_e4m3(kBM, kBNx);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t tl = 0;  // tiles done by this CTA
      bool ok = true;
      for (int L = blockIdx.x; L < sch.total && ok; L += gridDim.x, ++tl) {
        const Tile t = sch.decode(L);
        const int kbs = t.seg ? p.k_blocks1 : p.k_blocks0;
        if (!ptx::mbar_wait(tempty, (tl & 1) ^ 1, p.err)) {
          set_error(p.err, kDevTimeoutMma);
          break;
        }
        ptx::tc_fence_after();
        for (int kb = 0; kb < kbs; ++kb) {
          if (!ptx::mbar_wait(&full[stage], phase, p.err) || !ptx::mbar_wait(&sfull[stage], phase, p.err)) {
            set_error(p.err, kDevTimeoutMma);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sfa = tmem_base + kSfCol + stage * kSfSlot;
          const uint32_t sfb = sfa + 4;
          const uint32_t sf_smem = ptx::smem_u32(sSF + stage * kSfBytes);
          ptx::tmem_cp_32x128b_x4(sfa, ptx::smem_desc_rows16(sf_smem));
          ptx::tmem_cp_32x128b_x4(sfb, ptx::smem_desc_rows16(sf_smem + kSfaBytes));
          ptx::tmem_cp_32x128b_x4(sfb + 4, ptx::smem_desc_rows16(sf_smem + kSfaBytes + 512));
          const uint64_t adesc = ptx::smem_desc_sw128(ptx::smem_u32(sA + stage * kABytesX));
          const uint64_t bdesc = ptx::smem_desc_sw128(ptx::smem_u32(sB + stage * kBBytesX));
#pragma unroll
          for (int k = 0; k < kBKx / kUKx; ++k)
            ptx::mma_mx_f8(tmem_base, adesc + 2 * k, bdesc + 2 * k, idesc, sfa, sfb, (kb | k) != 0);
          ptx::tc_commit(&empty[stage]);
          if (++stage == kStagesX) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) ptx::tc_commit(tfull);
      }
      ptx::tc_commit(mma_done);
      if (!ptx::mbar_wait(mma_done, 0, nullptr)) set_error(p.err, kDevTimeoutDrain);
    }
  } else if (warp == 2) {
    // ================= scale producer: a batch of four stages is loaded one
    // batch ahead of the batch being written out, so that the global loads
    // of a batch overlap the MMAs of the previous one.
    Cursor ld{(int)blockIdx.x, 0, 0, Tile{}};
    cursor_load_tile(ld, sch, p);
    Cursor wr = ld;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    float a0[4][4], b0[4][2], a1[4][4], b1[4][2];
    auto load_batch = [&](float (&a)[4][4], float (&b)[4][2]) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (ld.L < sch.total) {
          load_stage_scales<EPI>(p, ld.t, ld.kb, lane, a[j], b[j]);
          cursor_next(ld, sch, p);
        }
      }
    };
    auto write_batch = [&](float (&a)[4][4], float (&b)[4][2]) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (!ok || wr.L >= sch.total) return;
        if (!ptx::mbar_wait(&empty[stage], phase ^ 1, p.err)) {
          set_error(p.err, kDevTimeoutProducer);
          ok = false;
          return;
        }
        uint8_t* sf = sSF + stage * kSfBytes;
        uint4 wa;
        wa.x = ue8m0_byte(a[j][0]) * 0x01010101u;
        wa.y = ue8m0_byte(a[j][1]) * 0x01010101u;
        wa.z = ue8m0_byte(a[j][2]) * 0x01010101u;
        wa.w = ue8m0_byte(a[j][3]) * 0x01010101u;
        reinterpret_cast<uint4*>(sf)[lane] = wa;
        const uint32_t g0 = ue8m0_byte(b[j][0]) * 0x01010101u;
        const uint32_t g1 = ue8m0_byte(b[j][1]) * 0x01010101u;
        // B rows 32c + lane, c = 0..7 (SwiGLU: rows 0..63 / 128..191 gate, 64..127 / 192..255 up)
        const uint4 lo = (EPI == Fp8Epi::kSwiGLU) ? make_uint4(g0, g0, g1, g1) : make_uint4(g0, g0, g0, g0);
        const uint4 hi = (EPI == Fp8Epi::kSwiGLU) ? make_uint4(g0, g0, g1, g1) : make_uint4(g1, g1, g1, g1);
        reinterpret_cast<uint4*>(sf + kSfaBytes)[lane] = lo;
        reinterpret_cast<uint4*>(sf + kSfaBytes + 512)[lane] = hi;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sfull[stage]);
        cursor_next(wr, sch, p);
        if (++stage == kStagesX) {
          stage = 0;
          phase ^= 1;
        }
      }
    };
    load_batch(a0, b0);
    while (ok && wr.L < sch.total) {
      load_batch(a1, b1);
      write_batch(a0, b0);
      if (!ok || wr.L >= sch.total) break;
      load_batch(a0, b0);
      write_batch(a1, b1);
    }
  } else {
    // ================= epilogue (warps 3..10)
    const int q = warp & 3;
    const int half = (warp - 3) >> 2;
    const int r_in_tile = 32 * q + lane;
    uint32_t tl = 0;
    bool ok = true;
    for (int L = blockIdx.x; L < sch.total; L += gridDim.x, ++tl) {
      const Tile t = sch.decode(L);
      const int row = t.row0 + r_in_tile;
      const int rows_total = t.seg ? p.rows1 : p.rows_total0;
      const bool valid = row < t.row_end;
      if (ok && !ptx::mbar_wait(tfull, tl & 1, p.err)) {
        set_error(p.err, kDevTimeoutEpilogue);
        ok = false;
      }
      ptx::tc_fence_after();
      float acc[128];
      if (ok) {
        // four loads in flight at once, then one wait: the accumulator goes
        // back to the MMA warp after a single TMEM round trip
        const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16) + half * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld32_nowait(tb + c * 32, acc + 32 * c);
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_wait_ld(acc + 32 * c);
      } else {
#pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
      }
      // the accumulator is in registers: hand TMEM back to the MMA warp
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(tempty);
      if constexpr (EPI == Fp8Epi::kSwiGLU) {
        // h = silu(gate) * up for this half's 64 intermediate columns, then the
        // 1x128 e4m3 tile (power-of-two scale) shared with the other half
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          acc[j] = silu_fast(acc[j]) * acc[64 + j];
          amax = fmaxf(amax, fabsf(acc[j]));
        }
        s_amax[half * 128 + r_in_tile] = amax;
        epi_bar_x();
        amax = fmaxf(amax, s_amax[(half ^ 1) * 128 + r_in_tile]);
        epi_bar_x();  // s_amax is rewritten by the next tile
        const float scale = e4m3_tile_scale(amax, true);
        const float inv = __fdiv_rn(1.0f, scale);  // exact: scale is a power of two
        // the row's 64 codes, out through the warp's staging block
        uint4 w[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float* a = acc + 16 * v;
          w[v].x = pack4_e4m3_x(a[0] * inv, a[1] * inv, a[2] * inv, a[3] * inv);
          w[v].y = pack4_e4m3_x(a[4] * inv, a[5] * inv, a[6] * inv, a[7] * inv);
          w[v].z = pack4_e4m3_x(a[8] * inv, a[9] * inv, a[10] * inv, a[11] * inv);
          w[v].w = pack4_e4m3_x(a[12] * inv, a[13] * inv, a[14] * inv, a[15] * inv);
        }
        {
          uint8_t* out = static_cast<uint8_t*>(t.seg ? p.out1 : p.out0);
          const int ldo = t.seg ? p.ldo1 : p.ldo0;
          const int rbase = t.row0 + 32 * q;
          const int nrows = ok ? max(0, min(32, t.row_end - rbase)) : 0;
          warp_store_rows64(s_stage_out + (warp - 3) * kStgWarp, lane, w,
                            out + (size_t)rbase * ldo + t.n * 128 + half * 64, (size_t)ldo, nrows);
        }
        if (valid && ok && half == 0) {
          float* hs = t.seg ? p.out_scale1 : p.out_scale0;
          hs[(size_t)t.n * rows_total + row] = scale;
        }
      } else if constexpr (EPI == Fp8Epi::kCombine) {
        if (valid && ok) {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(t.seg ? p.out1 : p.out0);
          const int ldo = t.seg ? p.ldo1 : p.ldo0;
          const size_t o = (size_t)row * ldo + t.n * kBNx + half * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            add_bf16x32(acc + 32 * c, p.radd + o + 32 * c, 1.0f);
            store_bf16x32(out + o + 32 * c, acc + 32 * c);
          }
        }
      } else {
        // bf16 rows, 32 columns at a time through the warp's staging block
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(t.seg ? p.out1 : p.out0);
        const int ldo = t.seg ? p.ldo1 : p.ldo0;
        const int rbase = t.row0 + 32 * q;
        const int nrows = ok ? max(0, min(32, t.row_end - rbase)) : 0;
        uint8_t* base = reinterpret_cast<uint8_t*>(out + (size_t)rbase * ldo + t.n * kBNx + half * 128);
        uint8_t* stg = s_stage_out + (warp - 3) * kStgWarp;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
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
cudaError_t launch_mx_one(const Fp8GemmLaunch& L) {
  auto kern = tc_gemm_mx_kernel<EPI>;
  static int attr_done[64] = {};
  cudaError_t e = set_smem_once(kern, kSmemX, attr_done);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, kThreadsX, kSmemX, L.stream>>>(L.a0, L.b0, L.a1, L.b1, L.p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mx_gemm(const Fp8GemmLaunch& L) {
  if (L.p.groups0 > kMaxGroups) return cudaErrorInvalidValue;
  switch (L.epi) {
    case Fp8Epi::kSwiGLU: return launch_mx_one<Fp8Epi::kSwiGLU>(L);
    case Fp8Epi::kStore: return launch_mx_one<Fp8Epi::kStore>(L);
    case Fp8Epi::kCombine: return launch_mx_one<Fp8Epi::kCombine>(L);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
