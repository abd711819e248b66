// Stage 3 of the MoE layer, compute: the experts' SwiGLU FFNs as grouped GEMMs
// on the fifth-generation tensor cores (tcgen05, accumulators in tensor
// memory), operands staged by TMA, with the group shapes read on the device.
//
// Follows the compute stage of "Scalable Training of Mixture-of-Experts Models
// with Megatron Core" (es summary, Resumen técnico §2.1 step 3 and §2.3.C:
// many small expert GEMMs grouped into one kernel so the tensor cores stay
// busy; kernels read token counts from GPU memory, no host synchronisation).
// The backward keeps the page's W/D split (§2.3.B): data-gradient and
// weight-gradient GEMMs are separate launches.
//
// One persistent kernel family, one CTA per SM, 192 threads:
//   warp 0     TMA producer (one lane): A and B tiles into a STAGES-deep ring;
//   warp 1     MMA issuer (one lane) and tensor-memory owner;
//   warps 2-5  epilogue: tcgen05.ld of the 128 x BN fp32 accumulator, the
//              fused element-wise work, bf16 stores.
// Two accumulators live in tensor memory so the epilogue of one tile overlaps
// the main loop of the next.
//
// Two problem shapes:
//   row-grouped (forward and data gradients): group g owns rows
//     offsets[g] .. offsets[g]+counts[g]-1 of A and of the output, B is the
//     group's weight; tiles are 128 rows x BN columns inside the group;
//   K-grouped (weight gradients): the group's rows are the reduction
//     dimension; the output is the group's own [Mw x N] matrix.
// Every group segment is a multiple of 128 rows whose padding rows are zero,
// so no tile crosses into another group and no masking is needed.
#include "gemm_common.cuh"

namespace moe {
namespace gg {

// Drains one 128 x BN fp32 accumulator through the fused epilogue. This warp
// handles the accumulator rows q*32 .. q*32+31 (tensor-memory lane quarter q,
// lane = row within the quarter) starting at `tbase`.
//   mt: m-tile of the group (rows offsets[g] + 128*mt, or output rows 128*mt
//       of group g for weight gradients); nt: n-tile; nk: k-blocks accumulated
//       (0 = the accumulator was never written: weight gradients of empty groups).
template <int EPI, int BN>
__device__ __forceinline__ void epilogue_tile(const Params& p, const CUtensorMap* tmC,
                                              const CUtensorMap* tmC2, uint32_t tbase, int g,
                                              int mt, int nt, int nk, int q, int lane,
                                              const int* s_off, uint8_t* stage,
                                              uint32_t stage_u32) {
  const int row0 = p.kgrouped ? g * p.Mw + mt * BM + q * 32 : s_off[g] + mt * BM + q * 32;
  // rows of the stored tensor and of GU / h_out (these 32 rows share a 128-row block)
  const int orow = p.kgrouped ? row0 : page_row(p, kPageOut, row0);
  const int xrow = p.kgrouped ? row0 : page_row(p, kPageAux, row0);
  const int ncols = swiglu_fwd(EPI) ? BN / 2 : BN;
  const int f0 = swiglu_fwd(EPI) ? nt * (BN / 2) : nt * BN;
  // router term of this warp's row (lane) for the FC1 data gradient
  float rd = 0.f;
  const float* rw = nullptr;
  if (EPI == kEpiDgradRouter && g < p.router_E) {
    const int t = p.token_of[row0 + lane];
    if (t >= 0 && t < p.router_T) rd = p.dlogits[(long long)t * p.router_E + g];
    rw = p.W_r + (long long)g * p.N + f0;
  }
  if (EPI == kEpiStore || EPI == kEpiWgrad || EPI == kEpiDgradRouter || EPI == kEpiAddBf16) {
    // plain bf16 output in 32 x 64 boxes: 128-byte rows (128-byte swizzle), so
    // every store fills whole 128-byte lines; 64 accumulator columns per
    // tensor-memory wait
#pragma unroll 1
    for (int c = 0; c < ncols; c += 64) {
      uint32_t r0[32], r1[32];
      if (EPI == kEpiWgrad && nk == 0) {
#pragma unroll
        for (int i = 0; i < 32; ++i) r0[i] = r1[i] = 0u;
      } else {
        ptx::tmem_ld32(tbase + c, r0);
        ptx::tmem_ld32(tbase + c + 32, r1);
        ptx::tmem_ld_wait();
      }
      if (EPI == kEpiDgradRouter && rw) {
        // fp32 accumulator + dlogits * W_r, rounded to bf16 once
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 w4 = __ldg(reinterpret_cast<const float4*>(rw + c) + v);
          r0[4 * v] = __float_as_uint(fmaf(rd, w4.x, __uint_as_float(r0[4 * v])));
          r0[4 * v + 1] = __float_as_uint(fmaf(rd, w4.y, __uint_as_float(r0[4 * v + 1])));
          r0[4 * v + 2] = __float_as_uint(fmaf(rd, w4.z, __uint_as_float(r0[4 * v + 2])));
          r0[4 * v + 3] = __float_as_uint(fmaf(rd, w4.w, __uint_as_float(r0[4 * v + 3])));
          const float4 w5 = __ldg(reinterpret_cast<const float4*>(rw + c + 32) + v);
          r1[4 * v] = __float_as_uint(fmaf(rd, w5.x, __uint_as_float(r1[4 * v])));
          r1[4 * v + 1] = __float_as_uint(fmaf(rd, w5.y, __uint_as_float(r1[4 * v + 1])));
          r1[4 * v + 2] = __float_as_uint(fmaf(rd, w5.z, __uint_as_float(r1[4 * v + 2])));
          r1[4 * v + 3] = __float_as_uint(fmaf(rd, w5.w, __uint_as_float(r1[4 * v + 3])));
        }
      }
      if (EPI == kEpiAddBf16 && row0 + lane < p.dense_rows) {
        // fp32 accumulator + the bf16 value in place, rounded to bf16 once
        const uint4* src =
            reinterpret_cast<const uint4*>(p.aux + (long long)(row0 + lane) * p.ldaux + f0 + c);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          float f[8], f2[8];
          unpack8(__ldg(src + v), f);
          unpack8(__ldg(src + 4 + v), f2);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            r0[8 * v + i] = __float_as_uint(__uint_as_float(r0[8 * v + i]) + f[i]);
            r1[8 * v + i] = __float_as_uint(__uint_as_float(r1[8 * v + i]) + f2[i]);
          }
        }
      }
      uint4 o[4], o2[4];
      pack_slice(r0, o);
      pack_slice(r1, o2);
      // the staging box is free once TMA has read the previous one
      if (lane == 0) ptx::tma_store_wait_read();
      __syncwarp();
      uint8_t* rowp = stage + lane * 128;             // chunk j of row r at j ^ (r & 7)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) = o[j];
        *reinterpret_cast<uint4*>(rowp + (((j + 4) ^ (lane & 7)) << 4)) = o2[j];
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_2d(tmC, stage_u32, f0 + c, orow);
        ptx::tma_store_commit();
      }
    }
    return;
  }
  // routing weight of this warp's row (lane) and the row's partial <dh_s, h>
  // when the weight sits inside the expert
  constexpr bool WGT = EPI == kEpiSwigluFwdW || EPI == kEpiSwigluBwdW;
  const float rwt = WGT ? p.row_w[row0 + lane] : 1.f;
  float dot = 0.f;
  uint4 gq[4], uq[4];
  const __nv_bfloat16* gu = nullptr;
  if (swiglu_bwd(EPI)) {
    // G and U of the next 32 columns are loaded one slice ahead
    gu = p.aux + (long long)(xrow + lane) * p.ldaux;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      gq[v] = ldg_nc_v4(gu + f0 + v * 8);
      uq[v] = ldg_nc_v4(gu + p.F + f0 + v * 8);
    }
  }
#pragma unroll 1
  for (int c = 0; c < ncols; c += 32) {
    uint4 o0[4], o1[4], o2[4];
    if (swiglu_fwd(EPI)) {
      uint32_t rg[32], ru[32];
      ptx::tmem_ld32(tbase + c, rg);
      ptx::tmem_ld32(tbase + BN / 2 + c, ru);
      ptx::tmem_ld_wait();
      pack_slice(rg, o0);
      pack_slice(ru, o1);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        float gr[8], ur[8], hf[8];
        unpack8(o0[v], gr);
        unpack8(o1[v], ur);
#pragma unroll
        for (int i = 0; i < 8; ++i) hf[i] = WGT ? silu_f(gr[i]) * ur[i] * rwt : silu_f(gr[i]) * ur[i];
        o2[v] = pack8(hf);
      }
    } else if (swiglu_bwd(EPI)) {
      uint32_t r[32];
      ptx::tmem_ld32(tbase + c, r);
      uint4 gn[4], un[4];
      const int cn = (c + 32 < ncols) ? c + 32 : c;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        gn[v] = ldg_nc_v4(gu + f0 + cn + v * 8);
        un[v] = ldg_nc_v4(gu + p.F + f0 + cn + v * 8);
      }
      ptx::tmem_ld_wait();
      __nv_bfloat16* hrow =
          p.h_out ? p.h_out + (long long)(xrow + lane) * p.F + f0 + c : nullptr;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        if (WGT) swiglu_bwd8_w(r + v * 8, gq[v], uq[v], rwt, o0[v], o1[v], dot);
        else swiglu_bwd8(r + v * 8, gq[v], uq[v], o0[v], o1[v]);
        // fine-grained recompute: h of these columns from the stored G, U
        if (hrow) stg_v4(hrow + 8 * v, swiglu_h8<WGT>(gq[v], uq[v], rwt));
        gq[v] = gn[v];
        uq[v] = un[v];
      }
    } else if (EPI == kEpiStoreF32) {
      // fp32 output: one 32 x 32 box = 128-byte rows, 128-byte swizzle (chunk j
      // of row r at slot j ^ (r & 7))
      uint32_t r[32];
      ptx::tmem_ld32(tbase + c, r);
      ptx::tmem_ld_wait();
      if (lane == 0) ptx::tma_store_wait_read();
      __syncwarp();
      uint8_t* rowp = stage + lane * 128;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) =
            make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_2d(tmC, stage_u32, f0 + c, orow);
        ptx::tma_store_commit();
      }
      continue;
    }
    // the staging area is free once the previous boxes have been read by TMA
    if (lane == 0) ptx::tma_store_wait_read();
    __syncwarp();
    stage_row(stage, 0, lane, o0);
    stage_row(stage, 1, lane, o1);
    if (swiglu_fwd(EPI)) stage_row(stage, 2, lane, o2);
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (swiglu_fwd(EPI)) {
        ptx::tma_store_2d(tmC, stage_u32, f0 + c, orow);                      // G
        ptx::tma_store_2d(tmC, stage_u32 + kBoxBytes, p.F + f0 + c, orow);    // U
        ptx::tma_store_2d(tmC2, stage_u32 + 2 * kBoxBytes, f0 + c, orow);     // h
      } else {
        ptx::tma_store_2d(tmC, stage_u32, f0 + c, orow);                      // dG
        ptx::tma_store_2d(tmC, stage_u32 + kBoxBytes, p.F + f0 + c, orow);    // dU
      }
      ptx::tma_store_commit();
    }
  }
  if (EPI == kEpiSwigluBwdW) p.dw_part[(long long)(row0 + lane) * p.dw_nt + nt] = dot;
}

template <int EPI, int BN, int A_MN, int B_MN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2,
                    const Params p) {
  constexpr int BPARTS = b_parts<EPI>();
  using L = Layout<BN, STAGES, BPARTS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* ctrl = smem_raw + (base - raw) + L::TILES;
  const uint32_t ctrl_u = base + L::TILES;
  // control block: barriers, tensor-memory address, abort flag, tile tables
  const uint32_t bar_full = ctrl_u;                       // [STAGES]
  const uint32_t bar_empty = ctrl_u + 8 * STAGES;         // [STAGES]
  const uint32_t bar_tfull = ctrl_u + 16 * STAGES;        // [2]
  const uint32_t bar_tempty = ctrl_u + 16 * STAGES + 16;  // [2]
  const uint32_t bar_drain = ctrl_u + 16 * STAGES + 32;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 192);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 196);
  int* prefix = reinterpret_cast<int*>(ctrl + 256);       // [kMaxGroups+1]
  int* mtiles = reinterpret_cast<int*>(ctrl + 1344);      // [kMaxGroups]
  int* s_off = reinterpret_cast<int*>(ctrl + 2432);       // [kMaxGroups+1]
  int* s_cnt = reinterpret_cast<int*>(ctrl + 3520);       // [kMaxGroups]
  int* tmp = reinterpret_cast<int*>(ctrl + 4608);         // [33] scan scratch

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G;
  const int NT = swiglu_fwd(EPI) ? p.F / (BN / 2) : p.N / BN;
  for (int g = tid; g < G; g += kThreads) {
    const int c = p.chunk_rows > 0 ? min(p.chunk_rows, p.dense_rows - g * p.chunk_rows)
                  : p.dense_rows > 0 ? p.dense_rows : p.counts[g];
    s_cnt[g] = c;
    s_off[g] = p.chunk_rows > 0 ? g * p.chunk_rows : p.dense_rows > 0 ? 0 : p.offsets[g];
    const int mt = p.kgrouped ? p.Mw / BM : (c + BM - 1) / BM;
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
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar_full + 8 * s, 1);
      ptx::mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(bar_tfull + 8 * a, 1);
      ptx::mbar_init(bar_tempty + 8 * a, 128);
    }
    ptx::mbar_init(bar_drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), L::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (tid == 32 * 0) {
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
        const Tile t = decode(tile, prefix, mtiles, s_cnt, G, p.kgrouped, p.K, NT, p.n_fast);
        for (int kb = 0; kb < t.nk; ++kb) {
          if (!ptx::mbar_wait(bar_empty + 8 * stage, phase ^ 1u, kWaitBudget, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          ptx::mbar_arrive_expect_tx(fb, L::STAGE);
          const uint32_t sA = base + stage * L::STAGE;
          const uint32_t sB = sA + L::A_BYTES;
          const int k0 = kb * BK;
          if (A_MN == 0) {
            ptx::tma_load_2d(sA, &tmA, fb, k0, page_row(p, kPageA, s_off[t.g] + t.mt * BM));
          } else if constexpr (EPI != kEpiStoreF32) {
            // MN-major A: its two 64-column chunks in one request (chunked map)
            const int kr = page_row(p, kPageA, s_off[t.g] + k0);
            ptx::tma_load_3d(sA, &tmA, fb, 0, kr, t.mt * BM / 64);
          } else {
            const int kr = page_row(p, kPageA, s_off[t.g] + k0);
            ptx::tma_load_2d(sA, &tmA, fb, t.mt * BM, kr);
            ptx::tma_load_2d(sA + 8192, &tmA, fb, t.mt * BM + 64, kr);
          }
          if (swiglu_fwd(EPI)) {
            const int f0 = t.nt * (BN / 2);
            ptx::tma_load_2d(sB, &tmB, fb, k0, t.g * p.b_rows + f0);
            ptx::tma_load_2d(sB + (BN / 2) * 128, &tmB, fb, k0, t.g * p.b_rows + p.F + f0);
          } else if (B_MN == 0) {
#pragma unroll
            for (int q = 0; q < BPARTS; ++q)
              ptx::tma_load_2d(sB + q * L::B_BYTES, &tmB, fb, BPARTS * k0 + q * BK,
                               t.g * p.b_rows + t.nt * BN);
          } else if constexpr (EPI != kEpiStoreF32) {
            // MN-major B: its BN / 64 chunks in one request (chunked map)
            const int kr =
                p.kgrouped ? page_row(p, kPageB, s_off[t.g] + k0) : t.g * p.b_rows + k0;
            ptx::tma_load_3d(sB, &tmB, fb, 0, kr, t.nt * BN / 64);
          } else {
            // (the router's three-part B keeps the 2D map)
            const int kr =
                p.kgrouped ? page_row(p, kPageB, s_off[t.g] + k0) : t.g * p.b_rows + k0;
#pragma unroll
            for (int q = 0; q < BPARTS; ++q)
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                ptx::tma_load_2d(sB + q * L::B_BYTES + j * 8192, &tmB, fb, t.nt * BN + 64 * j,
                                 (int)(q * p.part_rows) + kr);
          }
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
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
      for (int s = 0; s < STAGES; ++s)
        if (issued_mask & (1u << s))
          ptx::mbar_wait(bar_full + 8 * s, (issued_phase >> s) & 1u, kWaitBudget, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = ptx::idesc_bf16(BM, BN, A_MN, B_MN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, issued = false;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const Tile t = decode(tile, prefix, mtiles, s_cnt, G, p.kgrouped, p.K, NT, p.n_fast);
        if (!ptx::mbar_wait(bar_tempty + 8 * acc, acc_phase ^ 1u, kWaitBudget, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < t.nk; ++kb) {
          if (!ptx::mbar_wait(bar_full + 8 * stage, phase, kWaitBudget, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sA = base + stage * L::STAGE;
          const uint32_t sB = sA + L::A_BYTES;
#pragma unroll
          for (int q = 0; q < BPARTS; ++q)
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = A_MN ? ptx::smem_desc_sw128(sA + kk * 2048, 8192, 1024)
                                       : ptx::smem_desc_sw128(sA + kk * 32, 16, 1024);
              const uint32_t sq = sB + q * L::B_BYTES;
              const uint64_t bd = B_MN ? ptx::smem_desc_sw128(sq + kk * 2048, 8192, 1024)
                                       : ptx::smem_desc_sw128(sq + kk * 32, 16, 1024);
              ptx::mma_bf16(d, ad, bd, IDESC, (kb | kk | q) ? 1u : 0u);
            }
          issued = true;
          ptx::mma_commit(bar_empty + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (t.nk > 0) ptx::mma_commit(bar_tfull + 8 * acc);
        else ptx::mbar_arrive(bar_tfull + 8 * acc);   // empty group: nothing to wait for
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
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
    const int q = warp & 3;                        // tensor-memory lane quarter
    uint8_t* stage = ctrl + kCtrlBytes + (warp - 2) * kStageBytes;
    const uint32_t stage_u32 = ctrl_u + kCtrlBytes + (warp - 2) * kStageBytes;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode(tile, prefix, mtiles, s_cnt, G, p.kgrouped, p.K, NT, p.n_fast);
      bool ok = ptx::mbar_wait(bar_tfull + 8 * acc, acc_phase, kWaitBudget, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) {
          record_status(p.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
      epilogue_tile<EPI, BN>(p, &tmC, &tmC2, tbase, t.g, t.mt, t.nt, t.nk, q, lane, s_off, stage,
                             stage_u32);
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar_tempty + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) ptx::tma_store_wait_all();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

// ------------------------------------------------------------ CTA-pair variant
// The same grouped GEMM with 256 x 256 tiles computed by a pair of CTAs on two
// SMs (a cluster of 2) with tcgen05.mma.cta_group::2: each CTA holds 128 rows
// of the A tile and 128 of the 256 B columns, so every SM streams 32 KB per
// 64-deep k-block instead of 48 KB for the same tensor work, and six stages
// fit in shared memory (five with the SwiGLU-backward ring below). Only the
// even CTA issues MMAs; both CTAs' TMA loads
// count on the even CTA's "full" barrier, the MMA completion is multicast to
// both CTAs, and both epilogues report back to the even CTA.
constexpr int kPairStage = 32768;                 // 16 KB of A + 16 KB of B per CTA

// SwiGLU-backward operand ring of the pair kernel: G and U of an epilogue
// warp's coming 32-column slices are brought into shared memory by TMA (a
// 32 x 32 box of each, the 64-byte swizzle of the output maps) two slices
// ahead of the slice being drained, across tile boundaries, so their DRAM
// latency hides behind the main loop; dG and dU are written back over G and U
// and stored by TMA from the same slot. Three slots per warp take the room of
// one operand stage (five stages instead of six).
constexpr int kGuSlots = 3;
constexpr int kGuSlotBytes = 2 * kBoxBytes;
constexpr int kGuRingBytes = kGuSlots * kGuSlotBytes;
constexpr int kGuBarOff = 4864;                   // ring mbarriers in the control block

template <int EPI>
struct PairCfg {
  static constexpr bool RING = swiglu_bwd(EPI);
  static constexpr int STAGES = RING ? 5 : 6;
  static constexpr int EPI_BYTES = RING ? kGuRingBytes : kStageBytes;   // per epilogue warp
  static constexpr int SMEM = STAGES * kPairStage + kCtrlBytes + 4 * EPI_BYTES + 1024;
};
static_assert(PairCfg<kEpiSwigluBwd>::SMEM <= 232448, "pair SwiGLU-bwd shared memory");
static_assert(PairCfg<kEpiStore>::SMEM <= 232448, "pair shared memory");
static_assert(kGuBarOff >= 4608 + 33 * 4 && kGuBarOff + 4 * kGuSlots * 8 <= kCtrlBytes,
              "ring barriers inside the control block, after the scan scratch");

// dG and dU of one 32-column slice from dH (fp32, 32 tensor-memory columns of
// this lane's row) and the row's G and U, in place in a ring slot: 16-byte
// chunk j of the row sits at slot j ^ ((row >> 1) & 3) of its 64 bytes.
template <bool WGT>
__device__ __forceinline__ void swiglu_bwd_slice_inplace(uint8_t* slot, int lane,
                                                         const uint32_t (&r)[32], float rwt,
                                                         float& dot, __nv_bfloat16* hrow) {
  uint8_t* grow = slot + lane * 64;
  uint8_t* urow = grow + kBoxBytes;
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int pos = (v ^ sw) << 4;
    uint4 dg, du;
    // fine-grained recompute: h of these 8 columns from the stored G, U
    if (hrow)
      stg_v4(hrow + 8 * v, swiglu_h8<WGT>(*reinterpret_cast<const uint4*>(grow + pos),
                                          *reinterpret_cast<const uint4*>(urow + pos), rwt));
    if (WGT)
      swiglu_bwd8_w(r + v * 8, *reinterpret_cast<const uint4*>(grow + pos),
                    *reinterpret_cast<const uint4*>(urow + pos), rwt, dg, du, dot);
    else
      swiglu_bwd8(r + v * 8, *reinterpret_cast<const uint4*>(grow + pos),
                  *reinterpret_cast<const uint4*>(urow + pos), dg, du);
    *reinterpret_cast<uint4*>(grow + pos) = dg;
    *reinterpret_cast<uint4*>(urow + pos) = du;
  }
}

template <int EPI, int A_MN, int B_MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmC,
                         const __grid_constant__ CUtensorMap tmC2, const Params p) {
  using PC = PairCfg<EPI>;
  constexpr int BN = 256, STAGES = PC::STAGES;
  constexpr int A_BYTES = 16384;
  constexpr uint32_t TMEM_COLS = 2 * BN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* ctrl = smem_raw + (base - raw) + STAGES * kPairStage;
  const uint32_t ctrl_u = base + STAGES * kPairStage;
  const uint32_t bar_full = ctrl_u;
  const uint32_t bar_empty = ctrl_u + 8 * STAGES;
  const uint32_t bar_tfull = ctrl_u + 16 * STAGES;
  const uint32_t bar_tempty = ctrl_u + 16 * STAGES + 16;
  const uint32_t bar_drain = ctrl_u + 16 * STAGES + 32;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 192);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 196);
  int* prefix = reinterpret_cast<int*>(ctrl + 256);
  int* mtiles = reinterpret_cast<int*>(ctrl + 1344);
  int* s_off = reinterpret_cast<int*>(ctrl + 2432);
  int* s_cnt = reinterpret_cast<int*>(ctrl + 3520);
  int* tmp = reinterpret_cast<int*>(ctrl + 4608);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const int G = p.G;
  const int NT = swiglu_fwd(EPI) ? p.F / (BN / 2) : p.N / BN;
  for (int g = tid; g < G; g += kThreads) {
    const int c = p.chunk_rows > 0 ? min(p.chunk_rows, p.dense_rows - g * p.chunk_rows)
                  : p.dense_rows > 0 ? p.dense_rows : p.counts[g];
    s_cnt[g] = c;
    s_off[g] = p.chunk_rows > 0 ? g * p.chunk_rows : p.dense_rows > 0 ? 0 : p.offsets[g];
    const int mt = p.kgrouped ? p.Mw / BM : (c + BM - 1) / BM;
    mtiles[g] = mt;
    prefix[g] = ((mt + 1) >> 1) * NT;              // pair tiles of the group
  }
  if (tid == 0) *abort_flag = 0;
  __syncthreads();
  const int total = block_exclusive_scan(prefix, G, tmp);
  if (tid == 0) prefix[G] = total;
  __syncthreads();
  if (cluster >= total) return;                    // both CTAs of the pair leave together

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar_full + 8 * s, 1);
      ptx::mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(bar_tfull + 8 * a, 1);
      ptx::mbar_init(bar_tempty + 8 * a, 8);       // 4 epilogue warps x 2 CTAs
    }
    ptx::mbar_init(bar_drain, 1);
    if (PC::RING)
      for (int i = 0; i < 4 * kGuSlots; ++i) ptx::mbar_init(ctrl_u + kGuBarOff + 8 * i, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  if (tid == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // pair tile -> (group, m-pair, n-tile); m-pairs fastest
  auto decode_pair = [&](int pt, int& g, int& mp, int& nt, int& nk) {
    g = find_group(prefix, G, pt);
    const int local = pt - prefix[g];
    const int npairs = (mtiles[g] + 1) >> 1;
    if (p.n_fast) {
      nt = local % NT;
      mp = local / NT;
    } else {
      mp = local % npairs;
      nt = local / npairs;
    }
    nk = p.kgrouped ? (s_cnt[g] + BK - 1) / BK : p.K / BK;
  };

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      uint32_t leader_full[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) leader_full[s] = ptx::mapa_shared(bar_full + 8 * s, 0);
      for (int pt = cluster; pt < total && ok; pt += nclusters) {
        int g, mp, nt, nk;
        decode_pair(pt, g, mp, nt, nk);
        const int mt = 2 * mp + (int)rank;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(bar_empty + 8 * stage, phase ^ 1u, kWaitBudget, abort_flag)) {
            ok = false;
            break;
          }
          if (rank == 0) ptx::mbar_arrive_expect_tx(bar_full + 8 * stage, 2 * kPairStage);
          const uint32_t fb = leader_full[stage];
          const uint32_t sA = base + stage * kPairStage;
          const uint32_t sB = sA + A_BYTES;
          const int k0 = kb * BK;
          if (A_MN == 0) {
            ptx::tma_load_2d_pair(sA, &tmA, fb, k0, page_row(p, kPageA, s_off[g] + mt * BM));
          } else {
            const int kr = page_row(p, kPageA, s_off[g] + k0);
            ptx::tma_load_3d_pair(sA, &tmA, fb, 0, kr, mt * BM / 64);      // two 64-column chunks
          }
          if (swiglu_fwd(EPI)) {
            // CTA 0 brings the 128 gate rows, CTA 1 the matching 128 up rows
            ptx::tma_load_2d_pair(sB, &tmB, fb, k0,
                                  g * p.b_rows + (rank ? p.F : 0) + nt * (BN / 2));
          } else if (B_MN == 0) {
            ptx::tma_load_2d_pair(sB, &tmB, fb, k0, g * p.b_rows + nt * BN + (int)rank * 128);
          } else {
            const int kr = p.kgrouped ? page_row(p, kPageB, s_off[g] + k0) : g * p.b_rows + k0;
            ptx::tma_load_3d_pair(sB, &tmB, fb, 0, kr, (nt * BN + (int)rank * 128) / 64);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        record_status(p.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        // loads already issued land within microseconds; give them time
        const long long t0 = clock64();
        while (clock64() - t0 < 200000) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t IDESC = ptx::idesc_bf16(2 * BM, BN, A_MN, B_MN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, issued = false;
      const uint32_t peer_tfull[2] = {ptx::mapa_shared(bar_tfull, 1),
                                      ptx::mapa_shared(bar_tfull + 8, 1)};
      for (int pt = cluster; pt < total && ok; pt += nclusters) {
        int g, mp, nt, nk;
        decode_pair(pt, g, mp, nt, nk);
        if (!ptx::mbar_wait(bar_tempty + 8 * acc, acc_phase ^ 1u, kWaitBudget, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(bar_full + 8 * stage, phase, kWaitBudget, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sA = base + stage * kPairStage;
          const uint32_t sB = sA + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? ptx::smem_desc_sw128(sA + kk * 2048, 8192, 1024)
                                     : ptx::smem_desc_sw128(sA + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? ptx::smem_desc_sw128(sB + kk * 2048, 8192, 1024)
                                     : ptx::smem_desc_sw128(sB + kk * 32, 16, 1024);
            ptx::mma_bf16_pair(d, ad, bd, IDESC, (kb | kk) ? 1u : 0u);
          }
          issued = true;
          ptx::mma_commit_pair(bar_empty + 8 * stage, 3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (nk > 0) {
          ptx::mma_commit_pair(bar_tfull + 8 * acc, 3);
        } else {                                   // empty group: nothing to wait for
          ptx::mbar_arrive(bar_tfull + 8 * acc);
          ptx::mbar_arrive_cluster(peer_tfull[acc]);
        }
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        record_status(p.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      if (issued) {
        ptx::mma_commit_pair(bar_drain, 1);
        ptx::mbar_wait(bar_drain, 0, kWaitBudget, nullptr);
      }
    }
  } else if constexpr (PC::RING) {
    // ------------------------------------------- SwiGLU-backward epilogue
    const int q = warp & 3, ew = warp - 2;
    uint8_t* ring = ctrl + kCtrlBytes + ew * kGuRingBytes;
    const uint32_t ring_u32 = ctrl_u + kCtrlBytes + ew * kGuRingBytes;
    const uint32_t rbar = ctrl_u + kGuBarOff + ew * 8 * kGuSlots;
    const uint32_t leader_tempty[2] = {ptx::mapa_shared(bar_tempty, 0),
                                       ptx::mapa_shared(bar_tempty + 8, 0)};
    // this CTA's rows of pair tile pt, or -1 for the odd tile of a group
    auto tile_rows = [&](int pt, int& row0, int& f0) {
      int g, mp, nt, nk;
      decode_pair(pt, g, mp, nt, nk);
      const int mt = 2 * mp + (int)rank;
      row0 = s_off[g] + mt * BM + q * 32;
      f0 = nt * BN;
      return mt < mtiles[g];
    };
    // load cursor: the next slice whose G and U are to be fetched
    int lpt = cluster, lc = 0, lrow = 0, lf0 = 0;
    while (lpt < total && !tile_rows(lpt, lrow, lf0)) lpt += nclusters;
    uint32_t issued = 0, used = 0;
    auto issue = [&]() {
      if (lpt >= total) return;
      const uint32_t slot = issued % kGuSlots;
      if (lane == 0) {
        const uint32_t b = rbar + 8 * slot, dst = ring_u32 + slot * kGuSlotBytes;
        ptx::mbar_arrive_expect_tx(b, kGuSlotBytes);
        const int grow = page_row(p, kPageAux, lrow);
        ptx::tma_load_2d(dst, &tmC2, b, lf0 + lc, grow);                  // G
        ptx::tma_load_2d(dst + kBoxBytes, &tmC2, b, p.F + lf0 + lc, grow);  // U
      }
      ++issued;
      lc += 32;
      if (lc == BN) {
        lc = 0;
        do lpt += nclusters;
        while (lpt < total && !tile_rows(lpt, lrow, lf0));
      }
    };
    issue();
    issue();
    uint32_t acc = 0, acc_phase = 0;
    bool ok = true;
    for (int pt = cluster; pt < total && ok; pt += nclusters) {
      int row0, f0;
      const bool mine = tile_rows(pt, row0, f0);
      ok = __all_sync(0xffffffffu,
                      ptx::mbar_wait(bar_tfull + 8 * acc, acc_phase, kWaitBudget, abort_flag));
      if (!ok) break;
      ptx::tc_fence_after();
      if (mine) {
        const uint32_t tbase = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
        constexpr bool WGT = EPI == kEpiSwigluBwdW;
        const float rwt = WGT ? p.row_w[row0 + lane] : 1.f;
        float dot = 0.f;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          const uint32_t slot = used % kGuSlots;
          ok = __all_sync(0xffffffffu, ptx::mbar_wait(rbar + 8 * slot, (used / kGuSlots) & 1u,
                                                      kWaitBudget, abort_flag));
          if (!ok) break;
          uint32_t r[32];
          ptx::tmem_ld32(tbase + c, r);
          ptx::tmem_ld_wait();
          swiglu_bwd_slice_inplace<WGT>(
              ring + slot * kGuSlotBytes, lane, r, rwt, dot,
              p.h_out ? p.h_out + (long long)(page_row(p, kPageAux, row0) + lane) * p.F + f0 + c
                      : nullptr);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const uint32_t src = ring_u32 + slot * kGuSlotBytes;
            const int orow = page_row(p, kPageOut, row0);
            ptx::tma_store_2d(&tmC, src, f0 + c, orow);                    // dG
            ptx::tma_store_2d(&tmC, src + kBoxBytes, p.F + f0 + c, orow);  // dU
            ptx::tma_store_commit();
            // the slot of the slice before this one is free once its stores have read it
            ptx::tma_store_wait_read_1();
          }
          ++used;
          issue();
        }
        if (!ok) break;
        if (WGT) p.dw_part[(long long)(row0 + lane) * p.dw_nt + f0 / BN] = dot;
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(leader_tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok) {
      if (lane == 0) {
        record_status(p.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // loads still in flight land before the CTA may exit
      for (; used < issued; ++used)
        ptx::mbar_wait(rbar + 8 * (used % kGuSlots), (used / kGuSlots) & 1u, kWaitBudget, nullptr);
    }
    if (lane == 0) ptx::tma_store_wait_all();
  } else {
    const int q = warp & 3;
    uint8_t* stage = ctrl + kCtrlBytes + (warp - 2) * kStageBytes;
    const uint32_t stage_u32 = ctrl_u + kCtrlBytes + (warp - 2) * kStageBytes;
    const uint32_t leader_tempty[2] = {ptx::mapa_shared(bar_tempty, 0),
                                       ptx::mapa_shared(bar_tempty + 8, 0)};
    uint32_t acc = 0, acc_phase = 0;
    for (int pt = cluster; pt < total; pt += nclusters) {
      int g, mp, nt, nk;
      decode_pair(pt, g, mp, nt, nk);
      bool ok = ptx::mbar_wait(bar_tfull + 8 * acc, acc_phase, kWaitBudget, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) {
          record_status(p.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      ptx::tc_fence_after();
      const int mt = 2 * mp + (int)rank;
      if (mt < mtiles[g]) {                        // the odd tile of a group has no partner rows
        const uint32_t tbase = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
        epilogue_tile<EPI, BN>(p, &tmC, &tmC2, tbase, g, mt, nt, nk, q, lane, s_off, stage,
                               stage_u32);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(leader_tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) ptx::tma_store_wait_all();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int EPI, int BN, int A_MN, int B_MN, int STAGES>
static cudaError_t run(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                       const CUtensorMap& c2, const Params& p, cudaStream_t s) {
  using L = Layout<BN, STAGES, b_parts<EPI>()>;
  static_assert(L::SMEM <= 232448, "shared memory per block");
  auto kern = grouped_gemm_kernel<EPI, BN, A_MN, B_MN, STAGES>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<num_sms(), kThreads, L::SMEM, s>>>(a, b, c, c2, p);
  return cudaGetLastError();
}

// CTA-pair launch: as many clusters as can be resident at once (the tile loop
// strides statically over clusters, so every launched cluster must run).
template <int EPI, int A_MN, int B_MN>
static cudaError_t run_pair(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                            const CUtensorMap& c2, const Params& p, cudaStream_t s) {
  auto kern = grouped_gemm_pair_kernel<EPI, A_MN, B_MN>;
  static int grid = 0;
  if (grid == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairCfg<EPI>::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = PairCfg<EPI>::SMEM;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &lc);
    if (e != cudaSuccess || clusters <= 0) {
      (void)cudaGetLastError();
      clusters = num_sms() / 2;
    }
    grid = 2 * clusters;
  }
  kern<<<grid, kThreads, PairCfg<EPI>::SMEM, s>>>(a, b, c, c2, p);
  return cudaGetLastError();
}

// CTA pairs (256-row tiles) for GEMMs whose output width is a multiple of 256
// and whose experts expect at least 512 rows each; otherwise the single-CTA
// kernel (128-row tiles). An expert's rows are padded to 128, and a pair tile
// that holds only one valid 128-row half still runs both halves, so with few
// rows per expert (about 256: fine-grained experts) pairs run up to twice the
// MMA work of the useful rows, and their weight-gradient tiles are short in K
// as well. Measured on the 256-expert, 8192-token shape: forward 5.95 -> 5.74
// ms and backward 14.3 -> 13.1 ms with single-CTA tiles; at 1024 rows per
// expert pairs are faster.
static bool use_pairs(const moe_config& c, int n) {
  const long long per_expert = c.capacity_factor > 0.f
                                   ? (long long)capacity_rows(c)
                                   : (long long)c.T * c.k / (c.E > 0 ? c.E : 1);
  return n % 256 == 0 && per_expert >= 512;
}

}  // namespace gg

using namespace gg;

// N tiles of the FC2 data gradient (F wide): 256-column tiles when F is a
// multiple of 256 (CTA pairs or single CTAs), else 128.
int dw_tiles(const moe_config& c) { return c.F % 256 == 0 ? c.F / 256 : c.F / 128; }

cudaError_t launch_ffn_fc1(const moe_config& c, const void* x_perm, const int32_t* counts,
                           const int32_t* offsets, const void* W13, void* GU, void* h,
                           int32_t* status, cudaStream_t s, const float* row_w,
                           const StashMap& sm) {
  const int64_t SR = stash_rows(c, sm);
  const int G = c.E + c.n_shared;
  CUtensorMap a, b, oc, oc2;
  if (!make_map(&a, x_perm, c.H, SR, 128) ||
      !make_map(&b, W13, c.H, (uint64_t)G * 2 * c.F, 128) ||
      !make_out_map(&oc, GU, 2ULL * c.F, SR) || !make_out_map(&oc2, h, c.F, SR))
    return cudaErrorInvalidValue;
  Params p = base_params(c, counts, offsets, status);
  p.pages = sm.pages;
  p.page_ops = sm.pages ? kPageA | kPageOut : 0;
  p.K = c.H;
  p.b_rows = 2 * c.F;
  p.out = static_cast<__nv_bfloat16*>(GU);
  p.ldo = 2LL * c.F;
  p.out2 = static_cast<__nv_bfloat16*>(h);
  p.ldo2 = c.F;
  if (row_w) {                                     // h_s = w_row silu(G) U
    p.row_w = row_w;
    if (use_pairs(c, 256)) return run_pair<kEpiSwigluFwdW, 0, 0>(a, b, oc, oc2, p, s);
    return run<kEpiSwigluFwdW, 256, 0, 0, 4>(a, b, oc, oc2, p, s);
  }
  if (use_pairs(c, 256)) return run_pair<kEpiSwigluFwd, 0, 0>(a, b, oc, oc2, p, s);
  return run<kEpiSwigluFwd, 256, 0, 0, 4>(a, b, oc, oc2, p, s);
}

cudaError_t launch_ffn_fc2(const moe_config& c, const void* h, const int32_t* counts,
                           const int32_t* offsets, const void* W2, void* y_perm,
                           int32_t* status, cudaStream_t s, const StashMap& sm) {
  const int64_t SR = stash_rows(c, sm);
  const int G = c.E + c.n_shared;
  const int bn = (c.H % 256 == 0) ? 256 : 128;
  const bool pair = use_pairs(c, c.H);
  CUtensorMap a, b, oc;
  if (!make_map(&a, h, c.F, SR, 128) ||
      !make_map(&b, W2, c.F, (uint64_t)G * c.H, pair ? 128 : bn) ||
      !make_out_map_w64(&oc, y_perm, c.H, SR))
    return cudaErrorInvalidValue;
  const CUtensorMap& oc2 = oc;
  Params p = base_params(c, counts, offsets, status);
  p.pages = sm.pages;
  p.page_ops = sm.pages ? kPageA | kPageOut : 0;
  p.N = c.H;
  p.K = c.F;
  p.b_rows = c.H;
  p.out = static_cast<__nv_bfloat16*>(y_perm);
  p.ldo = c.H;
  if (pair) return run_pair<kEpiStore, 0, 0>(a, b, oc, oc2, p, s);
  return bn == 256 ? run<kEpiStore, 256, 0, 0, 4>(a, b, oc, oc2, p, s)
                   : run<kEpiStore, 128, 0, 0, 6>(a, b, oc, oc2, p, s);
}

cudaError_t launch_ffn_fc2_dgrad(const moe_config& c, const void* dO_perm, const int32_t* counts,
                                 const int32_t* offsets, const void* W2, const void* GU,
                                 void* dGU, int32_t* status, cudaStream_t s, const float* row_w,
                                 float* dw_part, void* h_out, const StashMap& sm) {
  const int64_t R = rows_max(c);
  const int G = c.E + c.n_shared;
  const int bn = (c.F % 256 == 0) ? 256 : 128;
  CUtensorMap a, b, oc, gu;
  if (!make_map(&a, dO_perm, c.H, R, 128) ||
      !make_map_chunks(&b, W2, c.F, (uint64_t)G * c.H, use_pairs(c, c.F) ? 2 : bn / 64) ||
      !make_out_map(&oc, dGU, 2ULL * c.F, R) ||
      !make_out_map(&gu, GU, 2ULL * c.F, stash_rows(c, sm)))
    return cudaErrorInvalidValue;
  const CUtensorMap& oc2 = gu;    // the pair kernel loads G and U through this map
  Params p = base_params(c, counts, offsets, status);
  p.pages = sm.pages;
  p.page_ops = sm.pages ? kPageAux : 0;
  p.N = c.F;
  p.K = c.H;
  p.b_rows = c.H;
  p.out = static_cast<__nv_bfloat16*>(dGU);
  p.ldo = 2LL * c.F;
  p.aux = static_cast<const __nv_bfloat16*>(GU);
  p.ldaux = 2LL * c.F;
  p.h_out = static_cast<__nv_bfloat16*>(h_out);
  if (row_w) {                                     // dh = w_row dh_s, partial <dh_s, h>
    p.row_w = row_w;
    p.dw_part = dw_part;
    p.dw_nt = dw_tiles(c);
    if (use_pairs(c, c.F)) return run_pair<kEpiSwigluBwdW, 0, 1>(a, b, oc, oc2, p, s);
    return bn == 256 ? run<kEpiSwigluBwdW, 256, 0, 1, 4>(a, b, oc, oc2, p, s)
                     : run<kEpiSwigluBwdW, 128, 0, 1, 6>(a, b, oc, oc2, p, s);
  }
  if (use_pairs(c, c.F)) return run_pair<kEpiSwigluBwd, 0, 1>(a, b, oc, oc2, p, s);
  return bn == 256 ? run<kEpiSwigluBwd, 256, 0, 1, 4>(a, b, oc, oc2, p, s)
                   : run<kEpiSwigluBwd, 128, 0, 1, 6>(a, b, oc, oc2, p, s);
}

cudaError_t launch_ffn_fc1_dgrad(const moe_config& c, const void* dGU, const int32_t* counts,
                                 const int32_t* offsets, const void* W13, const int32_t* token_of,
                                 const float* dlogits, const float* W_r, void* dX_perm,
                                 int32_t* status, cudaStream_t s) {
  const int64_t R = rows_max(c);
  const int G = c.E + c.n_shared;
  const int bn = (c.H % 256 == 0) ? 256 : 128;
  CUtensorMap a, b, oc;
  if (!make_map(&a, dGU, 2ULL * c.F, R, 128) ||
      !make_map_chunks(&b, W13, c.H, (uint64_t)G * 2 * c.F, use_pairs(c, c.H) ? 2 : bn / 64) ||
      !make_out_map_w64(&oc, dX_perm, c.H, R))
    return cudaErrorInvalidValue;
  const CUtensorMap& oc2 = oc;
  Params p = base_params(c, counts, offsets, status);
  p.N = c.H;
  p.K = 2 * c.F;
  p.b_rows = 2 * c.F;
  p.out = static_cast<__nv_bfloat16*>(dX_perm);
  p.ldo = c.H;
  p.token_of = token_of;
  p.dlogits = dlogits;
  p.W_r = W_r;
  p.router_E = c.E;
  p.router_T = c.T;
  if (use_pairs(c, c.H)) return run_pair<kEpiDgradRouter, 0, 1>(a, b, oc, oc2, p, s);
  return bn == 256 ? run<kEpiDgradRouter, 256, 0, 1, 4>(a, b, oc, oc2, p, s)
                   : run<kEpiDgradRouter, 128, 0, 1, 6>(a, b, oc, oc2, p, s);
}

cudaError_t launch_ffn_wgrad_fc2(const moe_config& c, const void* dO_perm, const void* h,
                                 const int32_t* counts, const int32_t* offsets, void* dW2,
                                 int32_t* status, cudaStream_t s, const StashMap& sm) {
  const int64_t R = rows_max(c);
  const int bn = (c.F % 256 == 0) ? 256 : 128;
  const int G = c.E + c.n_shared;
  CUtensorMap a, b, oc;
  if (!make_map_chunks(&a, dO_perm, c.H, R, 2) ||
      !make_map_chunks(&b, h, c.F, stash_rows(c, sm), use_pairs(c, c.F) ? 2 : bn / 64) ||
      !make_out_map_w64(&oc, dW2, c.F, (uint64_t)G * c.H))
    return cudaErrorInvalidValue;
  const CUtensorMap& oc2 = oc;
  Params p = base_params(c, counts, offsets, status);
  p.pages = sm.pages;
  p.page_ops = sm.pages ? kPageB : 0;
  p.kgrouped = 1;
  p.Mw = c.H;
  p.N = c.F;
  p.out = static_cast<__nv_bfloat16*>(dW2);
  p.ldo = c.F;
  p.out_gstride = (long long)c.H * c.F;
  p.n_fast = 1;                 // see launch_ffn_wgrad_fc1
  if (use_pairs(c, c.F)) return run_pair<kEpiWgrad, 1, 1>(a, b, oc, oc2, p, s);
  return bn == 256 ? run<kEpiWgrad, 256, 1, 1, 4>(a, b, oc, oc2, p, s)
                   : run<kEpiWgrad, 128, 1, 1, 6>(a, b, oc, oc2, p, s);
}

cudaError_t launch_ffn_wgrad_fc1(const moe_config& c, const void* dGU, const void* x_perm,
                                 const int32_t* counts, const int32_t* offsets, void* dW13,
                                 int32_t* status, cudaStream_t s, const StashMap& sm) {
  const int64_t R = rows_max(c);
  const int bn = (c.H % 256 == 0) ? 256 : 128;
  const int G = c.E + c.n_shared;
  CUtensorMap a, b, oc;
  if (!make_map_chunks(&a, dGU, 2ULL * c.F, R, 2) ||
      !make_map_chunks(&b, x_perm, c.H, stash_rows(c, sm), use_pairs(c, c.H) ? 2 : bn / 64) ||
      !make_out_map_w64(&oc, dW13, c.H, (uint64_t)G * 2 * c.F))
    return cudaErrorInvalidValue;
  const CUtensorMap& oc2 = oc;
  Params p = base_params(c, counts, offsets, status);
  p.pages = sm.pages;
  p.page_ops = sm.pages ? kPageB : 0;
  p.kgrouped = 1;
  p.Mw = 2 * c.F;
  p.N = c.H;
  p.out = static_cast<__nv_bfloat16*>(dW13);
  p.ldo = c.H;
  p.out_gstride = 2LL * c.F * c.H;
  // tiles n-fastest: the clusters running at once share the A slice (the
  // expert's dGU columns) and write whole rows of dW13 (DeepSeek-V3-shaped
  // weight-gradient stage 6.97 -> 6.78 ms; Mixtral- and Qwen3-shaped unchanged)
  p.n_fast = 1;
  if (use_pairs(c, c.H)) return run_pair<kEpiWgrad, 1, 1>(a, b, oc, oc2, p, s);
  return bn == 256 ? run<kEpiWgrad, 256, 1, 1, 4>(a, b, oc, oc2, p, s)
                   : run<kEpiWgrad, 128, 1, 1, 6>(a, b, oc, oc2, p, s);
}

// Router logits on the tensor cores: logits[T,E] = sum over the three bf16
// parts of W_r (W_r = W_hi + W_mid + W_lo exactly) of x . part^T. W3 [E, 3H]
// holds the parts interleaved per 64-column k-block (hi, mid, lo of columns
// 64j..64j+63, then of the next 64); one pipeline stage carries x's k-block j
// and the three part blocks 3j..3j+2, so every x tile is loaded once. fp32
// accumulation, one dense group of T rows (rows past T read zeros and are not
// stored). Needs E % 128 == 0.
cudaError_t launch_router_logits_tc(const moe_config& c, const void* x, const void* W3,
                                    float* logits, int32_t* status, cudaStream_t s) {
  CUtensorMap a, b, oc;
  if (!make_map(&a, x, c.H, c.T, 128) || !make_map(&b, W3, 3ULL * c.H, c.E, 128) ||
      !make_out_map_f32(&oc, logits, c.E, c.T))
    return cudaErrorInvalidValue;
  Params p{};
  p.G = 1;
  p.dense_rows = c.T;
  p.N = c.E;
  p.K = c.H;
  p.status = status;
  return run<kEpiStoreF32, 128, 0, 0, 3>(a, b, oc, oc, p, s);
}

// Router weight gradient on the tensor cores (E % 128 == 0), as K-grouped
// GEMMs over chunks of `chunk` tokens: P[c] = x[chunk c]^T . dlogits[chunk c]
// (H x E, fp32, P stacked [NG * H, E]). dlogits is split exactly into three bf16
// parts stacked along the rows of D3 [3 * Tp, E] (part q at rows q * Tp, rows
// T..Tp-1 zero); each pipeline stage carries one x^T k-block (MN-major, straight
// from x [T, H]) and the three part blocks. A chunk's products accumulate on the
// tensor cores (at most `chunk` terms); the chunks are added in order in fp32 by
// the caller.
cudaError_t launch_router_wgrad_tc(const moe_config& c, const void* x, const void* D3,
                                   long long Tp, float* P, int chunk, int32_t* status,
                                   cudaStream_t s) {
  const int NG = (c.T + chunk - 1) / chunk;
  if (NG > kMaxGroups) return cudaErrorInvalidValue;
  CUtensorMap a, b, oc;
  if (!make_map(&a, x, c.H, c.T, 64) || !make_map(&b, D3, c.E, 3ULL * Tp, 64) ||
      !make_out_map_f32(&oc, P, c.E, (uint64_t)NG * c.H))
    return cudaErrorInvalidValue;
  Params p{};
  p.kgrouped = 1;
  p.G = NG;
  p.dense_rows = c.T;
  p.chunk_rows = chunk;
  p.part_rows = Tp;
  p.Mw = c.H;
  p.N = c.E;
  p.status = status;
  return run<kEpiStoreF32, 128, 1, 1, 3>(a, b, oc, oc, p, s);
}

// dx[T, H] (bf16, in place) += A3 . B3^T on the tensor cores, one dense group
// of T rows (rows past T read zeros and are not stored): A3 [T, K3] and B3
// [H, K3] bf16, both K-major. The epilogue adds the fp32 accumulator to the
// bf16 value of dx it replaces and rounds once.
cudaError_t launch_router_dx_tc(const moe_config& c, const void* A3, const void* B3, int K3,
                                void* dx, int32_t* status, cudaStream_t s) {
  const int bn = (c.H % 256 == 0) ? 256 : 128;
  CUtensorMap a, b, oc;
  if (!make_map(&a, A3, K3, c.T, 128) || !make_map(&b, B3, K3, c.H, bn) ||
      !make_out_map_w64(&oc, dx, c.H, c.T))
    return cudaErrorInvalidValue;
  Params p{};
  p.G = 1;
  p.dense_rows = c.T;
  p.N = c.H;
  p.K = K3;
  p.b_rows = c.H;
  p.out = static_cast<__nv_bfloat16*>(dx);
  p.ldo = c.H;
  p.aux = static_cast<const __nv_bfloat16*>(dx);
  p.ldaux = c.H;
  p.status = status;
  return bn == 256 ? run<kEpiAddBf16, 256, 0, 0, 4>(a, b, oc, oc, p, s)
                   : run<kEpiAddBf16, 128, 0, 0, 6>(a, b, oc, oc, p, s);
}

}  // namespace moe
