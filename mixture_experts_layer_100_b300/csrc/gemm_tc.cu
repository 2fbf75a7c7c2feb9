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
constexpr int kAuxBytes = 12288;
constexpr int kRingBytes = 196608;

// A tile is MH 128-row halves x BN columns: the halves share each staged B
// slice (one tcgen05.mma per half), so MH = 2 moves a third less operand data
// from L2 per flop than MH = 1 at BN = 256. Each half's accumulator takes BN
// TMEM columns; two accumulators (epilogue of tile i beside the main loop of
// tile i+1) when they fit in TMEM's 512 columns, else one.
// SPLIT: fp32 operands as tf32 pairs. A staged K slice is then 32 fp32 (one
// 128-byte swizzle row) and every operand tile has a high part and, right
// after it, a remainder part.
template <int BN, int MH, bool SPLIT = false>
struct Cfg {
  static constexpr int kParts = SPLIT ? 2 : 1;
  static constexpr int kBKE = SPLIT ? 32 : kBK;  // K elements per staged slice
  static constexpr int kAPart = MH * kBM * 128;
  static constexpr int kBPart = BN * 128;
  static constexpr int kABytes = kParts * kAPart;
  static constexpr int kBBytes = kParts * kBPart;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStagesRaw = kRingBytes / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  static constexpr int kAccs = (2 * MH * BN <= 512) ? 2 : 1;
  static constexpr int kCols = kAccs * MH * BN;
  static constexpr int kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  static constexpr int kEpiWarps = 4 * MH;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kAuxBytes + kEpiWarps * kRowStageBytes;
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(!SPLIT || MH == 1, "tf32 pairs use one-half tiles");
  static_assert(MH * BN * kAccs <= 512, "TMEM columns");
};

template <int BN, Epi EPI, int MH, bool SPLIT>
__global__ void __launch_bounds__(Cfg<BN, MH, SPLIT>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                   const TcGemmParams p) {
  using C = Cfg<BN, MH, SPLIT>;
  constexpr int S = C::kStages;
  constexpr int NA = C::kAccs;
  constexpr int BMT = MH * kBM;  // rows per tile
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
  int* s_end = s_off + (kMaxGroups + 1);  // stored rows' end per group (counts0)

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
      if (p.counts0 != nullptr) s_end[g] = o0 + min(p.counts0[g], o1 - o0);
      const int mt = (o1 - o0 + BMT - 1) / BMT;
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
  sch.end = p.counts0 != nullptr ? s_end : nullptr;
  sch.groups0 = p.groups0;
  sch.tiles0 = s_tp[p.groups0];
  sch.n_tiles0 = p.n_tiles0;
  sch.n_tiles1 = p.n_tiles1;
  sch.rows1 = p.rows1;
  sch.mt1 = (p.rows1 + BMT - 1) / BMT;
  sch.total = sch.tiles0 + sch.mt1 * p.n_tiles1;
  sch.bm = BMT;
  sch.super_row = kSuperRow / MH;
  if ((int)blockIdx.x >= sch.total) return;  // nothing to do: no TMEM taken

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], C::kEpiWarps);
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
          // the second half is loaded (and multiplied) only if it has rows
          const bool h1 = MH == 2 && t.row0 + kBM < t.row_end;
          ptx::mbar_arrive_expect_tx(&full[stage], C::kStageBytes - (MH == 2 && !h1 ? kBM * 128 : 0));
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          uint8_t* a_dst = sA + stage * C::kABytes;
          uint8_t* b_dst = sB + stage * C::kBBytes;
          const int k0 = kb * C::kBKE;
          if constexpr (SPLIT) {
            // A [rows, 2, K]: high part, then remainder
            ptx::tma_load_3d(a_dst, ma, &full[stage], k0, 0, t.row0);
            ptx::tma_load_3d(a_dst + C::kAPart, ma, &full[stage], k0, 1, t.row0);
          } else {
            ptx::tma_load_2d(a_dst, ma, &full[stage], k0, t.row0);
            if (h1) ptx::tma_load_2d(a_dst + kBM * 128, ma, &full[stage], k0, t.row0 + kBM);
          }
          if constexpr (EPI == Epi::kRouterSigmoid) {
            // router weights [E, d] (SPLIT: [E, 2, d]); tile n covers experts n*BN..
            if constexpr (SPLIT) {
              ptx::tma_load_3d(b_dst, mb, &full[stage], k0, 0, t.n * BN);
              ptx::tma_load_3d(b_dst + C::kBPart, mb, &full[stage], k0, 1, t.n * BN);
            } else {
              ptx::tma_load_2d(b_dst, mb, &full[stage], k0, t.n * BN);
            }
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
            if constexpr (SPLIT) {
              // W13 [groups, 2I, 2, d]
#pragma unroll
              for (int part = 0; part < 2; ++part) {
                uint8_t* bd = b_dst + part * C::kBPart;
                ptx::tma_load_4d(bd + 0 * 8192, mb, &full[stage], k0, part, nrow, e);
                ptx::tma_load_4d(bd + 1 * 8192, mb, &full[stage], k0, part, p.I + nrow, e);
                ptx::tma_load_4d(bd + 2 * 8192, mb, &full[stage], k0, part, nrow + 64, e);
                ptx::tma_load_4d(bd + 3 * 8192, mb, &full[stage], k0, part, p.I + nrow + 64, e);
              }
            } else {
              ptx::tma_load_3d(b_dst + 0 * 8192, mb, &full[stage], k0, nrow, e);
              ptx::tma_load_3d(b_dst + 1 * 8192, mb, &full[stage], k0, p.I + nrow, e);
              ptx::tma_load_3d(b_dst + 2 * 8192, mb, &full[stage], k0, nrow + 64, e);
              ptx::tma_load_3d(b_dst + 3 * 8192, mb, &full[stage], k0, p.I + nrow + 64, e);
            }
          } else {
            // down projection: B = W2 [groups, d, I] (SPLIT: [groups, d, 2, I]);
            // the shared segment concatenates its S experts along K.
            const int kk = t.seg == 0 ? k0 : k0 % p.I;
            const int gi = t.seg == 0 ? t.group : k0 / p.I;
            if constexpr (SPLIT) {
              ptx::tma_load_4d(b_dst, mb, &full[stage], kk, 0, t.n * BN, gi);
              ptx::tma_load_4d(b_dst + C::kBPart, mb, &full[stage], kk, 1, t.n * BN, gi);
            } else {
              ptx::tma_load_3d(b_dst, mb, &full[stage], kk, t.n * BN, gi);
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
      constexpr uint32_t idesc = SPLIT ? ptx::idesc_tf32(kBM, BN) : ptx::idesc_bf16(kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int L = blockIdx.x; L < sch.total && ok; L += gridDim.x, ++it) {
        const Tile t = sch.decode(L);
        const int kbs = t.seg ? p.k_blocks1 : p.k_blocks0;
        const int acc = it % NA;
        if (!ptx::mbar_wait(&tempty[acc], ((it / NA) & 1) ^ 1, p.err)) {
          set_error(p.err, kDevTimeoutMma);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * MH * BN;
        const bool h1 = MH == 2 && t.row0 + kBM < t.row_end;
        for (int kb = 0; kb < kbs; ++kb) {
          if (!ptx::mbar_wait(&full[stage], phase, p.err)) {
            set_error(p.err, kDevTimeoutMma);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t adesc = ptx::smem_desc_sw128(ptx::smem_u32(sA + stage * C::kABytes));
          const uint64_t bdesc = ptx::smem_desc_sw128(ptx::smem_u32(sB + stage * C::kBBytes));
          if constexpr (SPLIT) {
            // three tf32 products per 8-wide K step (+32 bytes = +2 in the
            // 16-byte address field): hi*hi, hi*lo, lo*hi
            constexpr uint64_t a_lo = C::kAPart >> 4, b_lo = C::kBPart >> 4;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              ptx::mma_tf32(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
              ptx::mma_tf32(d_tmem, adesc + 2 * k, bdesc + b_lo + 2 * k, idesc, 1);
              ptx::mma_tf32(d_tmem, adesc + a_lo + 2 * k, bdesc + 2 * k, idesc, 1);
            }
          } else {
#pragma unroll
            for (int k = 0; k < kBK / kUK; ++k) {
              // +32 bytes along K per step = +2 in the 16-byte address field
              ptx::mma_f16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
            }
          }
          if (h1) {
            // second half: A rows 128..255 of the stage (+16 KB = +1024 in
            // the 16-byte address field), accumulator BN columns further
#pragma unroll
            for (int k = 0; k < kBK / kUK; ++k)
              ptx::mma_f16(d_tmem + BN, adesc + 1024 + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
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
    // ================= epilogue (warps 2 .. 2 + 4 MH - 1; warp w drains
    // half (w - 2) / 4, TMEM lane quarter w % 4)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;
    int it = 0;
    for (int L = blockIdx.x; L < sch.total; L += gridDim.x, ++it) {
      const Tile t = sch.decode(L);
      const int acc = it % NA;
      if (!ptx::mbar_wait(&tfull[acc], (it / NA) & 1, p.err)) {
        set_error(p.err, kDevTimeoutEpilogue);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + (acc * MH + half) * BN;
      const int rbase = t.row0 + half * kBM + 32 * q;
      const int row = rbase + lane;
      const bool valid = row < t.row_end;
      const int nrows = max(0, min(32, t.row_end - rbase));
      tile_epilogue<BN, EPI, SPLIT>(p, t, tbase, row, valid, aux + kAuxBytes + (warp - 2) * kRowStageBytes, rbase,
                                    nrows);
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

template <int BN, Epi EPI, int MH, bool SPLIT>
cudaError_t launch_one(const TcGemmLaunch& L) {
  auto kern = tc_gemm_kernel<BN, EPI, MH, SPLIT>;
  constexpr int smem = Cfg<BN, MH, SPLIT>::kSmemBytes;
  static int attr_done[64] = {};
  cudaError_t e = set_smem_once(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, Cfg<BN, MH, SPLIT>::kThreads, smem, L.stream>>>(L.a0, L.b0, L.a1, L.b1, L.p);
  return cudaGetLastError();
}

// One-half tiles, bf16 or tf32 pairs (router).
template <int BN, Epi EPI>
cudaError_t launch_1(const TcGemmLaunch& L) {
  return L.split ? launch_one<BN, EPI, 1, true>(L) : launch_one<BN, EPI, 1, false>(L);
}

// Expert GEMM launch: tf32 pairs on one-half tiles, or bf16 on one or two
// 128-row halves per tile (L.mh).
template <int BN, Epi EPI>
cudaError_t launch_mh(const TcGemmLaunch& L) {
  if (L.split) return launch_one<BN, EPI, 1, true>(L);
  return L.mh == 2 ? launch_one<BN, EPI, 2, false>(L) : launch_one<BN, EPI, 1, false>(L);
}

}  // namespace

cudaError_t launch_tc_gemm(const TcGemmLaunch& L) {
  if (L.p.groups0 > kMaxGroups) return cudaErrorInvalidValue;
  switch (L.epi) {
    case Epi::kRouterSigmoid:
      switch (L.bn) {
        case 32: return launch_1<32, Epi::kRouterSigmoid>(L);
        case 64: return launch_1<64, Epi::kRouterSigmoid>(L);
        case 128: return launch_1<128, Epi::kRouterSigmoid>(L);
        case 256: return launch_1<256, Epi::kRouterSigmoid>(L);
      }
      break;
    case Epi::kSwiGLU:
      if (L.bn == 256) return launch_mh<256, Epi::kSwiGLU>(L);
      break;
    case Epi::kStore:
      if (L.bn == 256) return launch_mh<256, Epi::kStore>(L);
      if (L.bn == 128) return launch_mh<128, Epi::kStore>(L);
      break;
    case Epi::kCombine:
      if (L.bn == 256) return launch_mh<256, Epi::kCombine>(L);
      if (L.bn == 128) return launch_mh<128, Epi::kCombine>(L);
      break;
    case Epi::kStoreF32:
      if (L.bn == 256) return launch_mh<256, Epi::kStoreF32>(L);
      if (L.bn == 128) return launch_mh<128, Epi::kStoreF32>(L);
      break;
    case Epi::kScatterAdd:
      if (L.bn == 256) return launch_mh<256, Epi::kScatterAdd>(L);
      if (L.bn == 128) return launch_mh<128, Epi::kScatterAdd>(L);
      break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
