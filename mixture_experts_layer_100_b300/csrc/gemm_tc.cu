// tcgen05 persistent grouped GEMM (bf16 x bf16 -> fp32 TMEM) with the MoE
// epilogues: router sigmoid, SwiGLU, plain store, and the fused combine.
#include "gemm_epi.cuh"
#include "gemm_sched.cuh"
#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBK = 64;           // bf16 elements per 128-byte swizzle row
constexpr int kUK = 16;           // K per tcgen05.mma (kind::f16)
constexpr int kThreads = 192;     // 6 warps
constexpr int kAuxBytes = 8192;
constexpr int kRingBytes = 196608;

template <int BN>
struct Cfg {
  static constexpr int kABytes = kBM * 128;
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStagesRaw = kRingBytes / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  static constexpr int kTmemCols = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                   : (2 * BN <= 256) ? 256 : 512;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kAuxBytes + 4 * kRowStageBytes;
};

template <int BN, Epi EPI>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                   const TcGemmParams p) {
  using C = Cfg<BN>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * C::kABytes;
  uint8_t* aux = smem + S * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(aux);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* s_tp = reinterpret_cast<int*>(aux + 256);
  int* s_mt = s_tp + (kMaxGroups + 1);
  int* s_off = s_mt + kMaxGroups;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- schedule: m-tiles per group and the first tile of each group
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
  if ((int)blockIdx.x >= sch.total) return;  // nothing to do: no TMEM taken

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 4);
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
    ptx::tmem_alloc(tmem_slot, C::kTmemCols);
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
      uint32_t phase = 0;
      uint32_t armed = 0;  // bit s: stage s has been armed at least once
      uint32_t armed_parity = 0;
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
          ptx::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          uint8_t* a_dst = sA + stage * C::kABytes;
          uint8_t* b_dst = sB + stage * C::kBBytes;
          const int k0 = kb * kBK;
          ptx::tma_load_2d(a_dst, ma, &full[stage], k0, t.row0);
          if constexpr (EPI == Epi::kRouterSigmoid) {
            ptx::tma_load_2d(b_dst, mb, &full[stage], k0, 0);
          } else if constexpr (EPI == Epi::kSwiGLU) {
            // B tile rows: [gate 0..63 | up 0..63 | gate 64..127 | up 64..127]
            // of the 128 intermediate columns this tile produces.
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
            // down projection: B = W2 [groups, d, I]; the shared segment
            // concatenates its S experts along K.
            if (t.seg == 0) {
              ptx::tma_load_3d(b_dst, mb, &full[stage], k0, t.n * BN, t.group);
            } else {
              ptx::tma_load_3d(b_dst, mb, &full[stage], k0 % p.I, t.n * BN, k0 / p.I);
            }
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Before leaving, make sure no copy is still landing in shared memory.
      for (int s = 0; s < S; ++s) {
        if (armed & (1u << s)) {
          if (!ptx::mbar_wait(&full[s], (armed_parity >> s) & 1u, nullptr)) {
            set_error(p.err, kDevTimeoutDrain);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16(kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < sch.total && ok; L += gridDim.x, ++it) {
        const Tile t = sch.decode(L);
        const int kbs = t.seg ? p.k_blocks1 : p.k_blocks0;
        const int acc = it & 1;
        if (!ptx::mbar_wait(&tempty[acc], ((it >> 1) & 1) ^ 1, p.err)) {
          set_error(p.err, kDevTimeoutMma);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < kbs; ++kb) {
          if (!ptx::mbar_wait(&full[stage], phase, p.err)) {
            set_error(p.err, kDevTimeoutMma);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t adesc = ptx::smem_desc_sw128(ptx::smem_u32(sA + stage * C::kABytes));
          const uint64_t bdesc = ptx::smem_desc_sw128(ptx::smem_u32(sB + stage * C::kBBytes));
#pragma unroll
          for (int k = 0; k < kBK / kUK; ++k) {
            // +32 bytes along K per step = +2 in the 16-byte address field
            ptx::mma_f16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
          }
          ptx::tc_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) ptx::tc_commit(&tfull[acc]);
      }
      // all issued MMAs complete before TMEM is released
      ptx::tc_commit(mma_done);
      if (!ptx::mbar_wait(mma_done, 0, nullptr)) set_error(p.err, kDevTimeoutDrain);
    }
  } else {
    // ================= epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int it = 0;
    for (int L = blockIdx.x; L < sch.total; L += gridDim.x, ++it) {
      const Tile t = sch.decode(L);
      const int acc = it & 1;
      if (!ptx::mbar_wait(&tfull[acc], (it >> 1) & 1, p.err)) {
        set_error(p.err, kDevTimeoutEpilogue);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + acc * BN;
      const int rbase = t.row0 + 32 * q;
      const int row = rbase + lane;
      const bool valid = row < t.row_end;
      const int nrows = max(0, min(32, t.row_end - rbase));
      tile_epilogue<BN, EPI>(p, t, tbase, row, valid, aux + kAuxBytes + (warp - 2) * kRowStageBytes, rbase, nrows);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
    }
  }

  __syncwarp();  // reconverge the role warps before the block barrier
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int BN, Epi EPI>
cudaError_t launch_one(const TcGemmLaunch& L) {
  auto kern = tc_gemm_kernel<BN, EPI>;
  constexpr int smem = Cfg<BN>::kSmemBytes;
  static int attr_done[64] = {};
  cudaError_t e = set_smem_once(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, kThreads, smem, L.stream>>>(L.a0, L.b0, L.a1, L.b1, L.p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_gemm(const TcGemmLaunch& L) {
  if (L.p.groups0 > kMaxGroups) return cudaErrorInvalidValue;
  switch (L.epi) {
    case Epi::kRouterSigmoid:
      switch (L.bn) {
        case 32: return launch_one<32, Epi::kRouterSigmoid>(L);
        case 64: return launch_one<64, Epi::kRouterSigmoid>(L);
        case 128: return launch_one<128, Epi::kRouterSigmoid>(L);
        case 256: return launch_one<256, Epi::kRouterSigmoid>(L);
      }
      break;
    case Epi::kSwiGLU:
      if (L.bn == 256) return launch_one<256, Epi::kSwiGLU>(L);
      break;
    case Epi::kStore:
      if (L.bn == 256) return launch_one<256, Epi::kStore>(L);
      if (L.bn == 128) return launch_one<128, Epi::kStore>(L);
      break;
    case Epi::kCombine:
      if (L.bn == 256) return launch_one<256, Epi::kCombine>(L);
      if (L.bn == 128) return launch_one<128, Epi::kCombine>(L);
      break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
