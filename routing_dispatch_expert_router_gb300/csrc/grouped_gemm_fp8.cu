// The expert GEMMs of the FP8 layer configuration on the block-scaled FP8
// tensor cores: tcgen05.mma.kind::mxf8f6f4 with E4M3 operands and UE8M0 block
// scales held in tensor memory.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (es
// summary, Resumen técnico §2.4) quantises the expert GEMMs to FP8 and names
// MXFP8 -- E4M3 values with power-of-two scales applied by the hardware -- as
// the Blackwell recipe. Here each 128 x 128 weight tile and each 1 x 128
// activation slice along K carries one UE8M0 scale; the MMA applies scales per
// 32-deep K slice (scale_vec::1X), so the four slices of a 128-wide K block
// read the same scale byte (fp8_layout.cuh). Products and fp32 accumulation
// happen in the tensor core; only the summation order differs from the fp64
// reference. The MXFP8 configuration (MX = 1) gives every 32-wide K slice its
// own scale (MX atom layout: one atom per 128-wide K block, the slice's byte
// picked by the MMA's scale-factor id).
//
// All six expert GEMMs: the row-grouped ones (forward FC1 + SwiGLU, FC2, the
// two data gradients; M = a group's rows, K = H or F) and the two weight
// gradients (K-grouped: M x N = the weight's shape, K = the group's rows, both
// operands read MN-major from their [rows, columns] buffers, quantised in
// 128 x 1 slices along the tokens).
//
// One persistent kernel per GEMM, one CTA per SM, 320 threads:
//   warp 0     TMA producer (one lane): per 128-deep k-block, A (128 rows) and
//              B (256 columns) E4M3 tiles plus three 512-byte scale atoms;
//   warp 1     MMA issuer (one lane) and tensor-memory owner: copies the
//              k-block's scale atoms into tensor memory (tcgen05.cp) and issues
//              four M=128 N=256 K=32 block-scaled MMAs;
//   warps 2-9  epilogue, two warps per tensor-memory lane quarter, 128 of the
//              256 accumulator columns each.
// Tensor memory: the 128 x 256 fp32 accumulator (columns 0-255) and one
// scale-factor slot of 16 columns per pipeline stage (A in the first 4, B in
// the next 8). Two accumulators would fill all 512 columns and leave no room
// for the scales, so there is one: the epilogue warps copy their 128 columns
// into registers and release the accumulator before they convert and store,
// which keeps the tensor cores idle only for the copy.
#include "fp8_layout.cuh"
#include "gemm_common.cuh"

namespace moe {
namespace gg {

constexpr int kF8Threads = 320;
constexpr int kF8MaxStages = 4;                   // size of the barrier arrays
constexpr int kF8BK = 128;                        // E4M3 elements (= bytes) per k-block
constexpr int kF8BN = 256;
constexpr int kF8ABytes = BM * kF8BK;             // 16 KB
constexpr int kF8BBytes = kF8BN * kF8BK;          // 32 KB
constexpr int kF8Stage = kF8ABytes + kF8BBytes;
constexpr int kF8SfStage = 3 * f8::kAtomBytes;    // A's atom, then B's two (128 columns each)
constexpr int kF8EpiWarps = 8;
// row maxima exchanged between the two epilogue warps of a lane quarter (the
// fused h quantisation: an h slice of 128 columns spans both warps), double
// buffered by tile parity: [2][4 quarters][2 warps][32 rows] fp32
constexpr int kF8XchBytes = 2 * 4 * 2 * 32 * 4;
constexpr int kF8XbarOff = 4864;                  // their 4 mbarriers in the control block
static_assert(kF8XbarOff >= 4608 + 33 * 4 && kF8XbarOff + 32 <= kCtrlBytes,
              "exchange barriers inside the control block, after the scan scratch");
constexpr uint32_t kF8TmemCols = 512;
constexpr uint32_t kF8SfCol = 256;                // first scale-factor column
constexpr uint32_t kF8SfSlotCols = 16;

// Shared-memory plan: four operand stages and a 32 x 32 bf16 output box (2 KB)
// per epilogue warp. (The weight gradients, whose tiles are a few 128-row K
// blocks deep, gain more from the fourth stage than from 32 x 64 boxes that
// write whole 128-byte lines: 7.52 -> 7.15 ms on the 256-expert FP8 layer.)
template <int EPI>
struct F8Cfg {
  static constexpr bool KG = EPI == kEpiWgrad;
  static constexpr int STAGES = 4;
  static constexpr int BOX = kBoxBytes;
  static constexpr int SF_OFF = STAGES * kF8Stage;
  static constexpr int CTRL_OFF = SF_OFF + STAGES * kF8SfStage;
  static constexpr int EPI_OFF = (CTRL_OFF + kCtrlBytes + 1023) / 1024 * 1024;
  static constexpr int XCH_OFF = EPI_OFF + kF8EpiWarps * BOX;
  static constexpr int SMEM = XCH_OFF + kF8XchBytes + 1024;
  static_assert(STAGES <= kF8MaxStages, "barrier arrays");
  static_assert(SMEM <= 232448, "FP8 grouped GEMM shared memory");
  static_assert(kF8SfCol + STAGES * kF8SfSlotCols <= kF8TmemCols, "FP8 tensor-memory columns");
};

// One 32 x 32 bf16 box (this warp's 32 rows, 32 columns) through the warp's
// staging slot to global memory by TMA.
__device__ __forceinline__ void f8_store_box(const CUtensorMap* tm, uint8_t* stage,
                                             uint32_t stage_u32, int lane, const uint4 (&v)[4],
                                             int c0, int c1) {
  if (lane == 0) ptx::tma_store_wait_read();       // the slot's previous box has been read
  __syncwarp();
  stage_row(stage, 0, lane, v);
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    ptx::tma_store_2d(tm, stage_u32, c0, c1);
    ptx::tma_store_commit();
  }
}

__device__ __forceinline__ const uint32_t (&slice32(const uint32_t (&r)[128], int i))[32] {
  return *reinterpret_cast<const uint32_t(*)[32]>(&r[32 * i]);
}

// The epilogue of one 128 x 256 tile once its accumulator columns are in
// registers (r: this warp's 32 rows x 128 columns, half = which 128): the
// SwiGLU forward with h's 1 x 128 E4M3 form (the two warps of a lane quarter
// exchange row maxima through `xch` under the mbarrier xbar + 8q), the SwiGLU
// backward (G, U of the first 32 columns already in gq, uq), the weight
// gradient's 32 x 32 boxes, or the plain / router-term store. Returns false
// when the exchange wait ran out (status recorded).
template <int EPI, int MX>
__device__ __forceinline__ bool f8_epilogue_tile(
    const Params& p, const CUtensorMap* tmC, const CUtensorMap* tmC2, uint8_t* stage,
    uint32_t stage_u32, float* xch, uint32_t xbar, volatile int* abort_flag, int g, int nt,
    int row0, int q, int half, int lane, uint32_t (&r)[128], const __nv_bfloat16* gu,
    uint4 (&gq)[4], uint4 (&uq)[4], int fb, uint32_t& x_phase) {
  // rows of the stored tensor and of h_out (a paged stash keeps these 32 rows in one page)
  const int orow = EPI == kEpiWgrad ? row0 : page_row(p, kPageOut, row0);
  const int xrow = EPI == kEpiWgrad ? row0 : page_row(p, kPageAux, row0);
  if (EPI == kEpiSwigluFwd) {
    const int f0 = nt * (kF8BN / 2) + 64 * half;
    uint4 ho[2][4];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint4 go[4], uo[4];
      pack_slice(slice32(r, c), go);
      pack_slice(slice32(r, 2 + c), uo);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        float gr[8], ur[8], hf[8];
        unpack8(go[v], gr);
        unpack8(uo[v], ur);
#pragma unroll
        for (int i = 0; i < 8; ++i) hf[i] = silu_f(gr[i]) * ur[i];
        ho[c][v] = pack8(hf);
      }
      f8_store_box(tmC, stage, stage_u32, lane, go, f0 + 32 * c, orow);          // G
      f8_store_box(tmC, stage, stage_u32, lane, uo, p.F + f0 + 32 * c, orow);    // U
      f8_store_box(tmC2, stage, stage_u32, lane, ho[c], f0 + 32 * c, orow);      // h
    }
    if (!MX && p.qout) {
      // h's 1 x 128 slice (columns nt*128 ..) is this warp's 64 columns and
      // its partner's: exchange the row maxima, then write the E4M3 codes
      float m = 0.f;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          float f[8];
          unpack8(ho[c][v], f);
          m = fmaxf(m, amax8(f));
        }
      float* xs = xch + ((x_phase * 4 + q) * 2) * 32;
      xs[half * 32 + lane] = m;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(xbar + 8 * q);
      const bool ok = __all_sync(
          0xffffffffu, ptx::mbar_wait(xbar + 8 * q, x_phase, kWaitBudget, abort_flag));
      if (!ok) {
        if (lane == 0) {
          record_status(p.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        return false;
      }
      const uint32_t code = ue8m0_code(fmaxf(m, xs[(half ^ 1) * 32 + lane]));
      const float inv = ue8m0_inv(code);
      const int row = row0 + lane;
      uint8_t* dst = p.qout + (size_t)row * p.F + f0;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint2 b[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          float f[8];
          unpack8(ho[c][v], f);
          b[v] = e4m3x8(f, inv);
        }
        *reinterpret_cast<uint4*>(dst + 32 * c) = make_uint4(b[0].x, b[0].y, b[1].x, b[1].y);
        *reinterpret_cast<uint4*>(dst + 32 * c + 16) = make_uint4(b[2].x, b[2].y, b[3].x, b[3].y);
      }
      if (half == 0)
        p.qsf[f8::atom_offset(row >> 7, nt, p.qsf_kg) + f8::atom_byte(row, nt)] =
            (uint8_t)code;
      x_phase ^= 1u;
    }
    if (MX && p.qout) {
      // h's 1 x 32 pieces (MXFP8): each is one of this thread's 32-column chunks
      const int row = row0 + lane;
      uint8_t* dst = p.qout + (size_t)row * p.F + f0;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float m = 0.f;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          float f[8];
          unpack8(ho[c][v], f);
          m = fmaxf(m, amax8(f));
        }
        const uint32_t code = ue8m0_code(m);
        const float inv = ue8m0_inv(code);
        uint2 b[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          float f[8];
          unpack8(ho[c][v], f);
          b[v] = e4m3x8(f, inv);
        }
        *reinterpret_cast<uint4*>(dst + 32 * c) = make_uint4(b[0].x, b[0].y, b[1].x, b[1].y);
        *reinterpret_cast<uint4*>(dst + 32 * c + 16) = make_uint4(b[2].x, b[2].y, b[3].x, b[3].y);
        const int col = f0 + 32 * c;
        p.qsf[f8::mx_atom_offset(row >> 7, col >> 7, p.qsf_kg) + f8::atom_byte(row, (col >> 5) & 3)] =
            (uint8_t)code;
      }
    }
  } else if (EPI == kEpiWgrad) {
    // dW rows g*Mw + m-tile.., columns n-tile*256 + 128*half.. in 32 x 32 boxes
    const int c0 = nt * kF8BN + 128 * half;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 o[4];
      pack_slice(slice32(r, c), o);
      f8_store_box(tmC, stage, stage_u32, lane, o, c0 + 32 * c, row0);
    }
  } else if (EPI == kEpiSwigluBwd) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 dg[4], du[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) swiglu_bwd8(&r[32 * c + 8 * v], gq[v], uq[v], dg[v], du[v]);
      if (p.h_out) {
        // fine-grained recompute: h of these 32 columns from the stored G, U
        __nv_bfloat16* hrow = p.h_out + (long long)(xrow + lane) * p.F + fb + 32 * c;
#pragma unroll
        for (int v = 0; v < 4; ++v) stg_v4(hrow + 8 * v, swiglu_h8<false>(gq[v], uq[v], 1.f));
      }
      if (c + 1 < 4) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          gq[v] = ldg_nc_v4(gu + fb + 32 * (c + 1) + v * 8);
          uq[v] = ldg_nc_v4(gu + p.F + fb + 32 * (c + 1) + v * 8);
        }
      }
      f8_store_box(tmC, stage, stage_u32, lane, dg, fb + 32 * c, orow);          // dG
      f8_store_box(tmC, stage, stage_u32, lane, du, p.F + fb + 32 * c, orow);    // dU
    }
  } else {
    // plain store (FC2) or FC1 data gradient plus the row's router term
    const int f0 = nt * kF8BN + 128 * half;
    float rd = 0.f;
    const float* rw = nullptr;
    if (EPI == kEpiDgradRouter && g < p.router_E) {
      const int tk = p.token_of[row0 + lane];
      if (tk >= 0 && tk < p.router_T) rd = p.dlogits[(long long)tk * p.router_E + g];
      rw = p.W_r + (long long)g * p.N + f0;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (EPI == kEpiDgradRouter && rw) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 w4 = __ldg(reinterpret_cast<const float4*>(rw + 32 * c) + v);
          float* a = reinterpret_cast<float*>(&r[32 * c + 4 * v]);
          a[0] = fmaf(rd, w4.x, a[0]);
          a[1] = fmaf(rd, w4.y, a[1]);
          a[2] = fmaf(rd, w4.z, a[2]);
          a[3] = fmaf(rd, w4.w, a[3]);
        }
      }
      uint4 o[4];
      pack_slice(slice32(r, c), o);
      f8_store_box(tmC, stage, stage_u32, lane, o, f0 + 32 * c, orow);
    }
  }
  return true;
}

template <int EPI, int B_MN, int MX>
__global__ void __launch_bounds__(kF8Threads, 1)
grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC,
                        const __grid_constant__ CUtensorMap tmC2, const Params p) {
  using C = F8Cfg<EPI>;
  constexpr int kStages = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t sf_u = base + C::SF_OFF;
  const uint32_t ctrl_u = base + C::CTRL_OFF;
  uint8_t* ctrl = sbase + C::CTRL_OFF;
  const uint32_t epi_u = base + C::EPI_OFF;
  uint8_t* epi = sbase + C::EPI_OFF;
  float* xch = reinterpret_cast<float*>(sbase + C::XCH_OFF);
  const uint32_t xbar = ctrl_u + kF8XbarOff;              // [4] quarters
  const uint32_t bar_full = ctrl_u;                       // [kStages]
  const uint32_t bar_empty = ctrl_u + 8 * kF8MaxStages;   // [kStages]
  const uint32_t bar_tfull = ctrl_u + 16 * kF8MaxStages;
  const uint32_t bar_tempty = bar_tfull + 8;
  const uint32_t bar_drain = bar_tfull + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 192);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 196);
  int* prefix = reinterpret_cast<int*>(ctrl + 256);
  int* mtiles = reinterpret_cast<int*>(ctrl + 1344);
  int* s_off = reinterpret_cast<int*>(ctrl + 2432);
  int* s_cnt = reinterpret_cast<int*>(ctrl + 3520);
  int* tmp = reinterpret_cast<int*>(ctrl + 4608);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G;
  const int NT = (EPI == kEpiSwigluFwd) ? p.F / (kF8BN / 2) : p.N / kF8BN;
  // k-blocks per tile: K / 128, or the group's row blocks (weight gradients)
  const int nk_fixed = C::KG ? 0 : p.K / kF8BK;
  const int n_fast = C::KG ? p.n_fast : 0;
  for (int g = tid; g < G; g += kF8Threads) {
    const int c = p.counts[g];
    s_cnt[g] = c;
    s_off[g] = p.offsets[g];
    const int mt = C::KG ? p.Mw / BM : (c + BM - 1) / BM;
    mtiles[g] = mt;
    prefix[g] = mt * NT;
  }
  if (tid == 0) *abort_flag = 0;
  __syncthreads();
  const int total = block_exclusive_scan(prefix, G, tmp);
  if (tid == 0) prefix[G] = total;
  __syncthreads();
  if ((int)blockIdx.x >= total) return;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar_full + 8 * s, 1);
      ptx::mbar_init(bar_empty + 8 * s, 1);
    }
    ptx::mbar_init(bar_tfull, 1);
    ptx::mbar_init(bar_tempty, kF8EpiWarps);
    ptx::mbar_init(bar_drain, 1);
    for (int qq = 0; qq < 4; ++qq) ptx::mbar_init(xbar + 8 * qq, 2);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kF8TmemCols);
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const Tile t = decode(tile, prefix, mtiles, s_cnt, G, 0, p.K, NT, n_fast);
        const int nk = C::KG ? (s_cnt[t.g] + kF8BK - 1) / kF8BK : nk_fixed;
        // A: rows row0.. (K-major), or columns m0.. of the group's rows k0..
        // (MN-major, weight gradients)
        const int row0 = C::KG ? t.mt * BM : s_off[t.g] + t.mt * BM;
        const int kr0 = C::KG ? s_off[t.g] : 0;
        // B: two 128-row (K-major) or 128-column (MN-major) boxes and their atoms
        int b0, b1, nb0, nb1;
        if (EPI == kEpiSwigluFwd) {
          const int f0 = t.nt * (kF8BN / 2);              // gate rows f0.., up rows F+f0..
          b0 = f0;
          b1 = p.F + f0;
        } else {
          b0 = t.nt * kF8BN;
          b1 = b0 + 128;
        }
        nb0 = b0 / 128;
        nb1 = b1 / 128;
        // atom rows: per group for the weights, shared by all groups for the
        // weight-gradient operands (their K blocks are the buffer's row blocks)
        const int64_t gb = C::KG ? 0 : (int64_t)t.g * p.sfb_nb;
        const uint8_t* sfa = p.sfa + (int64_t)(row0 / 128) * p.sfa_kg * f8::kAtomBytes;
        const uint8_t* sfb0 = p.sfb + (gb + nb0) * p.sfb_kg * f8::kAtomBytes;
        const uint8_t* sfb1 = p.sfb + (gb + nb1) * p.sfb_kg * f8::kAtomBytes;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(bar_empty + 8 * stage, phase ^ 1u, kWaitBudget, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          // the scale atoms travel only with the stages whose atoms the MMA
          // thread copies into tensor memory (every stage for MX; in the block
          // recipe a tile's first and every fourth K block of the operand)
          const bool with_sf = MX || kb == 0 || (((kr0 / kF8BK) + kb) & 3) == 0;
          ptx::mbar_arrive_expect_tx(fb, kF8Stage + (with_sf ? kF8SfStage : 0));
          const uint32_t sA = base + stage * kF8Stage;
          const uint32_t sB = sA + kF8ABytes;
          const int k0 = kr0 + kb * kF8BK;
          const int brow = C::KG ? k0 : t.g * p.b_rows + k0;
          if (C::KG) ptx::tma_load_2d(sA, &tmA, fb, row0, k0);
          else ptx::tma_load_2d(sA, &tmA, fb, k0, row0);
          if (B_MN == 0 && EPI != kEpiSwigluFwd) {
            // rows b0 .. b0 + 255 in one 256-row box (FC2's map)
            ptx::tma_load_2d(sB, &tmB, fb, k0, t.g * p.b_rows + b0);
          } else if (B_MN == 0) {
            ptx::tma_load_2d(sB, &tmB, fb, k0, t.g * p.b_rows + b0);
            ptx::tma_load_2d(sB + 16384, &tmB, fb, k0, t.g * p.b_rows + b1);
          } else {
            // MN-major: columns b0 .. b0 + 255 of rows brow.. as two 128-column
            // chunks in one request (the chunked 3D map)
            ptx::tma_load_3d(sB, &tmB, fb, 0, brow, b0 / 128);
          }
          const uint32_t sfs = sf_u + stage * kF8SfStage;
          // the atom of this K block: one per K block (MX) or per four
          const int64_t a4 = (int64_t)(MX ? k0 / kF8BK : k0 / kF8BK / f8::kAtomKBlocks) *
                             f8::kAtomBytes;
          if (with_sf) {
            ptx::bulk_load(sfs, sfa + a4, f8::kAtomBytes, fb);
            ptx::bulk_load(sfs + f8::kAtomBytes, sfb0 + a4, f8::kAtomBytes, fb);
            ptx::bulk_load(sfs + 2 * f8::kAtomBytes, sfb1 + a4, f8::kAtomBytes, fb);
          }
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        record_status(p.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // every load issued must land before the CTA may exit
      for (int s = 0; s < kStages; ++s)
        if (issued_mask & (1u << s))
          ptx::mbar_wait(bar_full + 8 * s, (issued_phase >> s) & 1u, kWaitBudget, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = ptx::idesc_mxf8_e4m3(BM, kF8BN, C::KG ? 1 : 0, B_MN);
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      uint32_t sf_slot = 0;                          // block recipe: current scale slot
      bool ok = true, issued = false;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        int nk = nk_fixed, kb0 = 0;
        if (C::KG) {
          // the group's row blocks; an empty group's tile takes no MMA (its
          // epilogue writes zeros without the accumulator)
          const Tile t = decode(tile, prefix, mtiles, s_cnt, G, 0, p.K, NT, n_fast);
          nk = (s_cnt[t.g] + kF8BK - 1) / kF8BK;
          kb0 = s_off[t.g] / kF8BK;
          if (nk == 0) continue;
        }
        if (!ptx::mbar_wait(bar_tempty, acc_phase ^ 1u, kWaitBudget, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(bar_full + 8 * stage, phase, kWaitBudget, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sfs = sf_u + stage * kF8SfStage;
          // scale atoms into tensor memory: MX has one per K block (a slot per
          // stage); in the block recipe an atom holds four consecutive K
          // blocks' scales, so it is copied when a tile starts and at every
          // fourth K block, into two alternating slots (the copies and the MMAs
          // of this thread run in issue order, so a slot is rewritten only
          // after the MMAs of the group before last)
          bool copy = true;
          uint32_t slot = stage;
          if (!MX) {
            copy = kb == 0 || ((kb0 + kb) & 3) == 0;
            if (copy) sf_slot ^= 1u;
            slot = sf_slot;
          }
          const uint32_t sfa_t = tmem_base + kF8SfCol + kF8SfSlotCols * slot;
          const uint32_t sfb_t = sfa_t + 4;
          if (copy) {
            ptx::tmem_cp_32x128b_warpx4(sfa_t, ptx::smem_desc_sf(sfs));
            ptx::tmem_cp_32x128b_warpx4(sfb_t, ptx::smem_desc_sf(sfs + f8::kAtomBytes));
            ptx::tmem_cp_32x128b_warpx4(sfb_t + 4, ptx::smem_desc_sf(sfs + 2 * f8::kAtomBytes));
          }
          // the scale byte inside the atom: this K block's (K blocks counted
          // from the start of the operand: the buffer's row blocks for the
          // weight gradients), or (MX) the 32-wide slice's
          const uint32_t idesc = ptx::idesc_with_sf_id(IDESC, (uint32_t)(kb0 + kb) & 3u);
          const uint32_t sA = base + stage * kF8Stage;
          const uint32_t sB = sA + kF8ABytes;
#pragma unroll
          for (int kk = 0; kk < kF8BK / 32; ++kk) {
            const uint64_t ad = C::KG ? ptx::smem_desc_sw128(sA + kk * 4096, 16384, 1024)
                                      : ptx::smem_desc_sw128(sA + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? ptx::smem_desc_sw128(sB + kk * 4096, 16384, 1024)
                                     : ptx::smem_desc_sw128(sB + kk * 32, 16, 1024);
            const uint32_t id = MX ? ptx::idesc_with_sf_id(IDESC, (uint32_t)kk) : idesc;
            ptx::mma_mxf8(tmem_base, ad, bd, id, sfa_t, sfb_t, (kb | kk) ? 1u : 0u);
          }
          issued = true;
          ptx::mma_commit(bar_empty + 8 * stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(bar_tfull);
        acc_phase ^= 1u;
      }
      if (!ok) {
        record_status(p.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // wait for every MMA issued by this thread before tensor memory is freed
      if (issued) {
        ptx::mma_commit(bar_drain);
        ptx::mbar_wait(bar_drain, 0, kWaitBudget, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // tensor-memory lane quarter
    const int half = (warp - 2) >> 2;             // which 128 accumulator columns
    uint8_t* stage = epi + (warp - 2) * C::BOX;
    const uint32_t stage_u32 = epi_u + (warp - 2) * C::BOX;
    const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16);
    uint32_t acc_phase = 0, x_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode(tile, prefix, mtiles, s_cnt, G, 0, p.K, NT, n_fast);
      const int row0 = C::KG ? t.g * p.Mw + t.mt * BM + q * 32 : s_off[t.g] + t.mt * BM + q * 32;
      // an empty group's weight-gradient tile: zeros, no accumulator
      const bool acc = !C::KG || s_cnt[t.g] > 0;
      // SwiGLU backward: G and U of the first 32 columns, loaded before the wait
      const __nv_bfloat16* gu = nullptr;
      uint4 gq[4], uq[4];
      int fb = 0;
      if (EPI == kEpiSwigluBwd) {
        fb = t.nt * kF8BN + 128 * half;
        gu = p.aux + (long long)(page_row(p, kPageAux, row0) + lane) * p.ldaux;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          gq[v] = ldg_nc_v4(gu + fb + v * 8);
          uq[v] = ldg_nc_v4(gu + p.F + fb + v * 8);
        }
      }
      uint32_t r[128];
      bool ok = true;
      if (acc) {
        ok = ptx::mbar_wait(bar_tfull, acc_phase, kWaitBudget, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (!ok) {
        if (lane == 0) {
          record_status(p.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      if (!acc) {
#pragma unroll
        for (int i = 0; i < 128; ++i) r[i] = 0u;
      } else {
        ptx::tc_fence_after();
        if (EPI == kEpiSwigluFwd) {
          // gate columns 64*half .. +63 and the matching up columns 128 + 64*half ..
          ptx::tmem_ld32(tq + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
          ptx::tmem_ld32(tq + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
          ptx::tmem_ld32(tq + 128 + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&r[64]));
          ptx::tmem_ld32(tq + 160 + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&r[96]));
        } else {
          ptx::tmem_ld128(tq + 128 * half, r);
        }
        ptx::tmem_ld_wait();
        // the accumulator is free for the next tile's MMAs
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_tempty);
        acc_phase ^= 1u;
      }

      if (!f8_epilogue_tile<EPI, MX>(p, &tmC, &tmC2, stage, stage_u32, xch, xbar, abort_flag, t.g,
                                     t.nt, row0, q, half, lane, r, gu, gq, uq, fb, x_phase))
        break;
    }
    if (lane == 0) ptx::tma_store_wait_all();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kF8TmemCols);
  }
}

template <int EPI, int B_MN, int MX>
static cudaError_t run_fp8_t(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                             const CUtensorMap& c2, const Params& p, cudaStream_t s) {
  auto kern = grouped_gemm_fp8_kernel<EPI, B_MN, MX>;
  constexpr int smem = F8Cfg<EPI>::SMEM;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<num_sms(), kF8Threads, smem, s>>>(a, b, c, c2, p);
  return cudaGetLastError();
}

template <int EPI, int B_MN>
static cudaError_t run_fp8(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                           const CUtensorMap& c2, const Params& p, bool mx, cudaStream_t s) {
  return mx ? run_fp8_t<EPI, B_MN, 1>(a, b, c, c2, p, s) : run_fp8_t<EPI, B_MN, 0>(a, b, c, c2, p, s);
}

static bool is_mx(const moe_config& c) { return c.dtype == MOE_DTYPE_MXFP8; }
// atoms per 128-row block of a K-long operand
static int sf_kg(const moe_config& c, int64_t K) { return (int)f8::sf_stride(K, is_mx(c)); }

}  // namespace gg

using namespace gg;

// FC1 + SwiGLU: GU = x_q W13_q^T (gate | up, bf16), h = bf16(silu(G) U), and
// h's 1-byte form (hq, hsf; 1 x 128 slices) for FC2.
cudaError_t launch_ffn_fc1_fp8(const moe_config& c, const uint8_t* xq, const uint8_t* xsf,
                               const int32_t* counts, const int32_t* offsets, const uint8_t* W13q,
                               const uint8_t* W13sf, void* GU, void* h, uint8_t* hq, uint8_t* hsf,
                               int32_t* status, cudaStream_t s, const StashMap& sm) {
  const int64_t R = rows_max(c), SR = stash_rows(c, sm);
  const int G = c.E + c.n_shared;
  CUtensorMap a, b, oc, oc2;
  if (!make_map_u8(&a, xq, c.H, R) || !make_map_u8(&b, W13q, c.H, (uint64_t)G * 2 * c.F) ||
      !make_out_map(&oc, GU, 2ULL * c.F, SR) || !make_out_map(&oc2, h, c.F, SR))
    return cudaErrorInvalidValue;
  Params p = base_params(c, counts, offsets, status);
  p.pages = sm.pages;
  p.page_ops = sm.pages ? kPageOut : 0;       // GU and h; x and h's 1-byte forms are not paged
  p.K = c.H;
  p.b_rows = 2 * c.F;
  p.sfa = xsf;
  p.sfa_kg = sf_kg(c, c.H);
  p.sfb = W13sf;
  p.sfb_nb = 2 * c.F / 128;
  p.sfb_kg = sf_kg(c, c.H);
  p.qout = hq;
  p.qsf = hsf;
  p.qsf_kg = sf_kg(c, c.F);
  return run_fp8<kEpiSwigluFwd, 0>(a, b, oc, oc2, p, is_mx(c), s);
}

// FC2: y_perm = h_q W2_q^T (bf16).
cudaError_t launch_ffn_fc2_fp8(const moe_config& c, const uint8_t* hq, const uint8_t* hsf,
                               const int32_t* counts, const int32_t* offsets, const uint8_t* W2q,
                               const uint8_t* W2sf, void* y_perm, int32_t* status,
                               cudaStream_t s, const StashMap& sm) {
  const int64_t R = rows_max(c);
  const int G = c.E + c.n_shared;
  CUtensorMap a, b, oc;
  // B: W2's rows of one 256-wide n-tile in a single box
  if (!make_map_u8(&a, hq, c.F, R) || !make_map_u8(&b, W2q, c.F, (uint64_t)G * c.H, 256) ||
      !make_out_map(&oc, y_perm, c.H, stash_rows(c, sm)))
    return cudaErrorInvalidValue;
  Params p = base_params(c, counts, offsets, status);
  p.pages = sm.pages;
  p.page_ops = sm.pages ? kPageOut : 0;
  p.N = c.H;
  p.K = c.F;
  p.b_rows = c.H;
  p.sfa = hsf;
  p.sfa_kg = sf_kg(c, c.F);
  p.sfb = W2sf;
  p.sfb_nb = c.H / 128;
  p.sfb_kg = sf_kg(c, c.F);
  return run_fp8<kEpiStore, 0>(a, b, oc, oc, p, is_mx(c), s);
}

// FC2 data gradient + SwiGLU backward: dh = dO_q W2_q (fp32, W2 read
// transposed: MN-major B), then dG, dU from the stored GU (bf16).
cudaError_t launch_ffn_fc2_dgrad_fp8(const moe_config& c, const uint8_t* dOq, const uint8_t* dOsf,
                                     const int32_t* counts, const int32_t* offsets,
                                     const uint8_t* W2q, const uint8_t* W2sf_t, const void* GU,
                                     void* dGU, int32_t* status, cudaStream_t s, void* h_out,
                                     const StashMap& sm) {
  const int64_t R = rows_max(c);
  const int G = c.E + c.n_shared;
  CUtensorMap a, b, oc;
  if (!make_map_u8(&a, dOq, c.H, R) || !make_map_u8_chunks(&b, W2q, c.F, (uint64_t)G * c.H, 2) ||
      !make_out_map(&oc, dGU, 2ULL * c.F, R))
    return cudaErrorInvalidValue;
  Params p = base_params(c, counts, offsets, status);
  p.pages = sm.pages;
  p.page_ops = sm.pages ? kPageAux : 0;       // GU and h_out
  p.N = c.F;
  p.K = c.H;
  p.b_rows = c.H;
  p.aux = static_cast<const __nv_bfloat16*>(GU);
  p.ldaux = 2LL * c.F;
  p.h_out = static_cast<__nv_bfloat16*>(h_out);
  p.sfa = dOsf;
  p.sfa_kg = sf_kg(c, c.H);
  p.sfb = W2sf_t;
  p.sfb_nb = c.F / 128;
  p.sfb_kg = sf_kg(c, c.H);
  return run_fp8<kEpiSwigluBwd, 1>(a, b, oc, oc, p, is_mx(c), s);
}

// FC1 data gradient: dX_perm = bf16(dGU_q W13_q + the row's router term)
// (W13 read transposed: MN-major B).
cudaError_t launch_ffn_fc1_dgrad_fp8(const moe_config& c, const uint8_t* dGq, const uint8_t* dGsf,
                                     const int32_t* counts, const int32_t* offsets,
                                     const uint8_t* W13q, const uint8_t* W13sf_t,
                                     const int32_t* token_of, const float* dlogits,
                                     const float* W_r, void* dX_perm, int32_t* status,
                                     cudaStream_t s) {
  const int64_t R = rows_max(c);
  const int G = c.E + c.n_shared;
  CUtensorMap a, b, oc;
  if (!make_map_u8(&a, dGq, 2ULL * c.F, R) ||
      !make_map_u8_chunks(&b, W13q, c.H, (uint64_t)G * 2 * c.F, 2) ||
      !make_out_map(&oc, dX_perm, c.H, R))
    return cudaErrorInvalidValue;
  Params p = base_params(c, counts, offsets, status);
  p.N = c.H;
  p.K = 2 * c.F;
  p.b_rows = 2 * c.F;
  p.token_of = token_of;
  p.dlogits = dlogits;
  p.W_r = W_r;
  p.router_E = c.E;
  p.router_T = c.T;
  p.sfa = dGsf;
  p.sfa_kg = sf_kg(c, 2LL * c.F);
  p.sfb = W13sf_t;
  p.sfb_nb = c.H / 128;
  p.sfb_kg = sf_kg(c, 2LL * c.F);
  return run_fp8<kEpiDgradRouter, 1>(a, b, oc, oc, p, is_mx(c), s);
}

// Weight gradients (K = each group's rows, both operands MN-major from their
// [rows, columns] buffers, 128 x 1 slices along the tokens):
// dW2[g] = dO_q^T h_q (M = H, N = F).
cudaError_t launch_ffn_wgrad_fc2_fp8(const moe_config& c, const uint8_t* dOq, const uint8_t* dOsf,
                                     const uint8_t* hq, const uint8_t* hsf, const int32_t* counts,
                                     const int32_t* offsets, void* dW2, int32_t* status,
                                     cudaStream_t s) {
  const int64_t R = rows_max(c);
  const int G = c.E + c.n_shared;
  CUtensorMap a, b, oc;
  if (!make_map_u8(&a, dOq, c.H, R) || !make_map_u8_chunks(&b, hq, c.F, R, 2) ||
      !make_out_map(&oc, dW2, c.F, (uint64_t)G * c.H))
    return cudaErrorInvalidValue;
  Params p = base_params(c, counts, offsets, status);
  p.Mw = c.H;
  p.N = c.F;
  p.K = 0;
  p.n_fast = 1;                 // see launch_ffn_wgrad_fc1_fp8
  p.sfa = dOsf;
  p.sfa_kg = sf_kg(c, R);
  p.sfb = hsf;
  p.sfb_kg = sf_kg(c, R);
  return run_fp8<kEpiWgrad, 1>(a, b, oc, oc, p, is_mx(c), s);
}

// dW13[g] = dGU_q^T x_q (M = 2F, N = H).
cudaError_t launch_ffn_wgrad_fc1_fp8(const moe_config& c, const uint8_t* dGq, const uint8_t* dGsf,
                                     const uint8_t* xq, const uint8_t* xsf, const int32_t* counts,
                                     const int32_t* offsets, void* dW13, int32_t* status,
                                     cudaStream_t s) {
  const int64_t R = rows_max(c);
  const int G = c.E + c.n_shared;
  CUtensorMap a, b, oc;
  if (!make_map_u8(&a, dGq, 2ULL * c.F, R) || !make_map_u8_chunks(&b, xq, c.H, R, 2) ||
      !make_out_map(&oc, dW13, c.H, (uint64_t)G * 2 * c.F))
    return cudaErrorInvalidValue;
  Params p = base_params(c, counts, offsets, status);
  p.Mw = 2 * c.F;
  p.N = c.H;
  p.K = 0;
  // tiles n-fastest: the CTAs running at once write whole rows of dW (full
  // 14 KB rows of dW13 rather than 512-byte pieces of every row), which HBM
  // takes faster (weight-gradient stage of the 256-expert FP8 layer 6.59 ->
  // 6.41 ms; dW2's order makes no difference)
  p.n_fast = 1;
  p.sfa = dGsf;
  p.sfa_kg = sf_kg(c, R);
  p.sfb = xsf;
  p.sfb_kg = sf_kg(c, R);
  return run_fp8<kEpiWgrad, 1>(a, b, oc, oc, p, is_mx(c), s);
}

}  // namespace moe
