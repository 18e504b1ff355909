// moe_tc.cu — the wide (prefill) calls on the 5th-generation tensor cores (tcgen05): the BF16
// router GEMM, the grouped NVFP4 expert GEMMs of the W4A4 and the W4A16/W4A8 paths, and the
// kernels that prepare their operands.
//
// Model card "Qwen3.8-Flash-Next NVIDIA NVFP4 for Infernix (bit-exact)", section "What is
// bit-exact and what is quantized": E2M1 codes with one E4M3 scale per 16 weights, an FP32
// multiplier and an FP32 activation input scale per matrix. The Infernix README, section
// "Activation precision", reads prompts in W4A4 on the FP4 tensor cores. Here that is
// tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (E2M1 x E2M1, UE4M3 scale per 16),
// 128 x 128 per instruction, K = 64, FP32 accumulators in tensor memory:
//
//   * tokens are grouped per expert into tiles of <= 128 slots ("token tiles"), laid out in a
//     padded permuted space (tile j = rows 128j..128j+127), so that a tile's activation codes
//     and scale-factor atoms are contiguous;
//   * the activation tile is the MMA's M side and the weight tile its N side, so the
//     accumulator is [slot][weight row] and one epilogue thread holds one slot's row;
//   * warp 0 issues TMA loads (tensor maps, 128-byte swizzle) of the weight and activation tiles
//     and bulk copies of the scale-factor atoms into a ring of stages guarded by mbarriers;
//     warp 1 copies the scale factors into tensor memory (tcgen05.cp) and issues the MMAs;
//     warps 2..9 are the epilogue (tensor memory -> registers, then SiLU*up and the NVFP4
//     quantisation of h, or the BF16 expert output Y);
//   * one thread issues all of a CTA's tensor-core instructions, and at these tile sizes that
//     issuing, not memory, bounds a CTA: the gate/up GEMM runs two CTAs per SM; the down GEMM
//     keeps a token tile's h in shared and tensor memory while it runs the expert's weight
//     tiles, and stores Y through TMA.
//
// Scale-factor atom (512 B, one K step of 64 for 128 rows): byte (r % 32) * 16 + (r / 32) * 4 + b
// holds the scale of row r, 16-element block b; tcgen05.cp.32x128b.warpx4 copies it into tensor
// memory in the layout the block-scaled MMA reads.
#include "moe_internal.cuh"

#include <cuda.h>
#include <cuda_bf16.h>

namespace moe {
namespace tc {

constexpr int kTileM = 128;
constexpr int kTileN = 128;
constexpr int kStageK = 256;                    // FP4 elements per stage = 128 bytes per row
constexpr int kTileBytes = kTileM * 128;        // 16 KB: one 128-row x 128-byte SW128 tile
constexpr int kSfStage = 4 * 512;               // 4 K steps of scale-factor atoms
constexpr int kStageBytes = 2 * kTileBytes + 2 * kSfStage;   // A, B, SFA, SFB = 36 KB
constexpr int kEpiWarps = 8;                    // two per tensor-memory lane quadrant
constexpr int kThreads = (2 + kEpiWarps) * 32;  // producer, MMA, epilogue warps
constexpr int kYStride = kTileM + 8;            // padded slot column of a transposed BF16 Y tile
constexpr int kTmemCols = 256;
constexpr int kSfCol = 128;                     // scale factors after the 128-column accumulator

// Shape of the two grouped FP4 GEMMs. A CTA runs one (token tile, weight tile) unit at a time and
// two CTAs share an SM: each CTA has one thread that issues the tensor-core instructions, and a
// single issuing thread spends about as long issuing a K step's 8 scale-factor copies and 4 MMAs
// as the tensor pipe takes to run them, so a second, independent issuer per SM is what keeps the
// pipe busy. That budget (half of an SM's shared and tensor memory) gives each CTA 3 stages of
// 36 KB and 256 tensor-memory columns: one 128-column accumulator and two sets of scale factors.
constexpr int kStages = 3;
constexpr int kCtasPerSm = 2;
constexpr int kSmem = kStages * kStageBytes + 1024;
static_assert(kCtasPerSm * (kSmem + 1024) <= 233472, "shared memory of two CTAs");
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kTileN >> 3) << 17) |
                            ((uint32_t)(kTileM >> 4) << 24);   // E2M1 x E2M1, UE4M3, 128x128

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Source descriptor of a 32-row x 16-byte scale-factor atom (rows 16 B apart, no swizzle).
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)(16 >> 4) << 16) |
         ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y,
                                       uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// TMA tensor store of a box from shared memory (bulk-group completion), and its group waits.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {   // sources of all groups read
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_but1() {  // all but the newest group read
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {        // all groups complete
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void mma_nvf4(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa,
                                         uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void epi_sync() {  // the epilogue warps
  asm volatile("bar.sync 2, %0;" ::"r"(kEpiWarps * 32) : "memory");
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

// Byte offset of (row r, 16-element block b) inside a scale-factor atom.
__device__ __forceinline__ int sf_atom_byte(int r, int b) {
  return (r & 31) * 16 + (r >> 5) * 4 + b;
}

struct TcParams {
  const uint8_t* sfa;    // weight scale-factor atoms (pack)
  const uint8_t* sfb;    // activation scale-factor atoms (workspace)
  const float* mult;     // [E][3]
  const float* dscale;   // [E] down input scale
  const float* dinv6;    // [E]
  float xS;              // activation input scale of gate/up
  int H, I, E;
  int MT;                // m tiles per token tile
  int nks;               // stages per tile
  int last_k4;           // K steps (of 64) in the last stage
  int a8;                // W4A16 kernels: 1 = W4A8 (E4M3 activations and h, per-matrix scales)
  int nsw;               // k_tc_down: weight-tile stages
  uint32_t ustride;      // k_tc_down: shared-memory bytes of one operand tile with its scales
};

// ------------------------------------------------------------------ shared pipeline skeleton
// Kernel body shared by gate/up and down: DOWN selects the operands, K and the epilogue. The MMA
// takes the activation tile as its M side and the weight tile as its N side, so that the
// accumulator is [slot][weight row]: one epilogue thread holds one slot's row, and for gate/up
// that row holds the 16 gate and 16 up values of each 16-element block of h side by side (the
// weight tile interleaves them by 16), so SiLU*up and the quantiser run inside one thread.
template <bool DOWN>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    k_tc_gemm(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
              const __grid_constant__ CUtensorMap tm_b, TcParams prm, WsView ws) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t full[kStages], empty[kStages], acc_full, acc_empty;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* smem = smem_raw + pad;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, kEpiWarps);
    fence_mbar_init();
    abort_s = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_s)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_s;
  pdl_wait();
  pdl_launch_dependents();

  const int NT = (int)ws.ctl[kCtlTokenTiles];
  const int ntiles = NT * prm.MT;
  const int H = prm.H, I = prm.I;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int it = 0;
      for (int t = blockIdx.x; t < ntiles && !abort_s; t += gridDim.x) {
        const int j = t / prm.MT, mt = t % prm.MT;
        const int e = __ldg(&ws.tt_expert[j]);
        for (int ks = 0; ks < prm.nks; ++ks, ++it) {
          const int s = it % kStages, n = it / kStages;
          if (n > 0 && !mbar_wait(&empty[s], (n - 1) & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
            break;
          }
          unsigned char* st = smem + s * kStageBytes;
          const int k4 = (ks == prm.nks - 1) ? prm.last_k4 : 4;
          mbar_arrive_expect_tx(&full[s], 2 * kTileBytes + 2 * 512 * k4);
          if (!DOWN) {
            // weight tile = the 64 gate and 64 up rows of intermediate tile mt, interleaved by 16
            // (tile rows 32q .. 32q+15: gate rows mt*64 + 16q .., 32q+16 .. 32q+31: the up rows of
            // the same indices)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              tma_2d(st + q * 4096, &tm_a0, ks * 128, e * I + mt * 64 + 16 * q, &full[s]);
              tma_2d(st + q * 4096 + 2048, &tm_a1, ks * 128, e * I + mt * 64 + 16 * q, &full[s]);
            }
          } else {
            tma_2d(st, &tm_a0, ks * 128, e * H + mt * 128, &full[s]);
          }
          tma_2d(st + kTileBytes, &tm_b, ks * 128, j * 128, &full[s]);
          const int katoms = DOWN ? I / 64 : H / 64;
          bulk_g2s(st + 2 * kTileBytes,
                   prm.sfa + (((size_t)e * prm.MT + mt) * katoms + 4 * ks) * 512, 512 * k4,
                   &full[s]);
          bulk_g2s(st + 2 * kTileBytes + kSfStage, prm.sfb + ((size_t)j * katoms + 4 * ks) * 512,
                   512 * k4, &full[s]);
        }
      }
      const int used = it < kStages ? it : kStages;
      for (int i = 0; i < used; ++i) {
        const int c = it - 1 - i;
        (void)mbar_wait(&full[c % kStages], (c / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int it = 0, tcount = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tcount) {
        // the accumulator of the previous unit has been read by the epilogue
        if (tcount > 0 && !abort_s && !mbar_wait(&acc_empty, (tcount - 1) & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        fence_after();
        for (int ks = 0; ks < prm.nks; ++ks, ++it) {
          const int s = it % kStages, n = it / kStages;
          if (!abort_s && !mbar_wait(&full[s], n & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
          }
          fence_after();
          unsigned char* st = smem + s * kStageBytes;
          const uint32_t w0 = smem_u32(st), x0 = smem_u32(st + kTileBytes);
          const uint32_t sfw0 = smem_u32(st + 2 * kTileBytes);
          const uint32_t sfx0 = smem_u32(st + 2 * kTileBytes + kSfStage);
          const uint32_t sfcol = tmem + kSfCol + (it & 1) * 32;
          const int k4 = (ks == prm.nks - 1) ? prm.last_k4 : 4;
          for (int q = 0; q < k4; ++q) {
            cp_sf(sfcol + 4 * q, desc_sf(sfx0 + q * 512));
            cp_sf(sfcol + 16 + 4 * q, desc_sf(sfw0 + q * 512));
          }
          for (int q = 0; q < k4; ++q) {
            mma_nvf4(tmem, desc_sw128(x0 + q * 32), desc_sw128(w0 + q * 32), sfcol + 4 * q,
                     sfcol + 16 + 4 * q, (ks > 0 || q > 0) ? 1u : 0u);
          }
          commit(&empty[s]);
        }
        commit(&acc_full);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..9)
    const int ew = warp - 2;              // epilogue warp 0..7
    const int quad = warp & 3;            // tensor-memory lanes 32*quad .. +31 (hardware rule)
    const int chalf = ew >> 2;            // columns 64*chalf .. +63 of the accumulator
    const int col = quad * 32 + lane;     // accumulator row = slot of the token tile
    int tcount = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tcount) {
      const int j = t / prm.MT, mt = t % prm.MT;
      // tile metadata (independent loads, issued before the wait)
      const int e = ws.tt_expert[j];
      const int slot0 = ws.tt_slot0[j], nval = ws.tt_n[j];
      if (!abort_s && !mbar_wait(&acc_full, tcount & 1)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
      }
      __syncwarp();
      fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16) + chalf * 64;
      uint32_t r0[32], r1[32];
      ld32(tbase, r0);
      ld32(tbase + 32, r1);
      // both halves are in registers: the accumulator goes back to the MMA warp
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty);
      if (col >= nval) continue;
      const size_t slot = (size_t)slot0 + col;
      if (!DOWN) {
        // columns 32q .. 32q+15: gate of the 16 indices mt*64 + 16q ..; 32q+16 .. 32q+31: up.
        // This thread's 64 columns are blocks q = 2*chalf, 2*chalf + 1 of the tile.
        const float mg = prm.mult[e * 3 + 0] * prm.xS, mu = prm.mult[e * 3 + 1] * prm.xS;
        const float Sd = prm.dscale[e], i6 = prm.dinv6[e];
        const size_t pslot = (size_t)j * 128 + col;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          float h[16];
          float a = 0.0f;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g = __uint_as_float(hb ? r1[i] : r0[i]) * mg;
            const float u = __uint_as_float(hb ? r1[16 + i] : r0[16 + i]) * mu;
            h[i] = (g / (1.0f + expf(-g))) * u;
            a = fmaxf(a, fabsf(h[i]));
          }
          const uint32_t sf = e4m3_encode_rn(__fmul_rn(a, i6));
          uint32_t lo = 0, hi = 0;
          if (sf != 0u) {
            const float rr = __frcp_rn(__fmul_rn(e4m3_value_nonneg(sf), Sd));
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              lo |= e2m1_encode_rn(__fmul_rn(h[i], rr)) << (4 * i);
              hi |= e2m1_encode_rn(__fmul_rn(h[8 + i], rr)) << (4 * i);
            }
          }
          const int ib = mt * 4 + chalf * 2 + hb;   // 16-element block of h along I
          *reinterpret_cast<uint2*>(ws.hq_perm + pslot * (I / 2) + ib * 8) = make_uint2(lo, hi);
          *reinterpret_cast<uint2*>(ws.hq + slot * (I / 2) + ib * 8) = make_uint2(lo, hi);
          ws.hsf_atoms[((size_t)j * (I / 64) + ib / 4) * 512 + sf_atom_byte(col, ib & 3)] =
              (uint8_t)sf;
          ws.hsf[slot * (I / 16) + ib] = (uint8_t)sf;
        }
      } else {
        // Y[slot][mt*128 + 64*chalf ..] = BF16(acc * md): 64 consecutive BF16 of one row, as
        // eight 16-byte stores
        const float md = prm.mult[e * 3 + 2] * prm.dscale[e];
        uint4* dst = reinterpret_cast<uint4*>(ws.y + slot * H + mt * 128 + chalf * 64);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i0 = (c * 8 + 2 * q) & 31;
            const uint32_t v0 = (c < 4) ? r0[i0] : r1[i0], v1 = (c < 4) ? r0[i0 + 1] : r1[i0 + 1];
            w[q] = (uint32_t)f32_to_bf16_rn(__uint_as_float(v0) * md) |
                   ((uint32_t)f32_to_bf16_rn(__uint_as_float(v1) * md) << 16);
          }
          dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

// ------------------------------------------------------------------ down GEMM, resident h
// Y[slot][row] = BF16(md * h[slot] . Wd[row]) for the W4A4 path when a token tile's h (K = I,
// up to 768) fits in shared memory twice. Each CTA (one per SM) takes token tiles j = CTA index,
// + grid, ... and runs the units (j, 128-row tile mt of H) of each for mt = 0 .. H/128 - 1, so the
// h tile of j and its scale factors (in tensor memory) stay in place while the CTA streams the
// expert's down-weight tiles; the next token tile's h loads into the other buffer meanwhile. Per
// unit only the weight tile and its scale factors move: half the copies of a unit that restages
// both operands. All CTAs sweep mt in the same order at about the same pace, so the CTAs holding
// token tiles of one expert read each of its weight tiles at about the same time, once from HBM
// and then from L2. The accumulators are double-buffered (two 128-column buffers), so the
// epilogue of one unit overlaps the next. Each epilogue warp writes its 32 slots' Y rows into its
// own 4 KB of shared memory (128-byte swizzled, conflict-free) and stores them with TMA, 32 or 16
// rows per box; the rows of a ragged tile past its last 16-row box go out as plain stores.
// Warp 0: TMA producer; warp 1: MMA issuer; warps 2..9: epilogue (as in k_tc_gemm<true>).
constexpr int kRhMaxStages = 6;
constexpr int kRhTmemCols = 512;
constexpr int kRhStaging = kEpiWarps * 32 * 128;   // 32 rows x 128 bytes per epilogue warp

__global__ void __launch_bounds__(kThreads, 1)
    k_tc_down(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
              const __grid_constant__ CUtensorMap tm_y32, const __grid_constant__ CUtensorMap tm_y16,
              TcParams prm, WsView ws) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t full[kRhMaxStages], empty[kRhMaxStages], h_full[2], h_empty[2], acc_full[2],
      acc_empty[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* smem = smem_raw + pad;
  const int nsw = prm.nsw;
  const uint32_t ustride = prm.ustride;
  const int nkc = prm.nks;                 // 128-byte K chunks of a row
  const int natoms = prm.I / 64;           // K steps of 64 = scale-factor atoms per tile
  const uint32_t ubytes = (uint32_t)nkc * kTileBytes + (uint32_t)natoms * 512;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < nsw; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&h_full[b], 1);
      mbar_init(&h_empty[b], 1);
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps);
    }
    fence_mbar_init();
    abort_s = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_s)),
                 "r"(kRhTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_s;
  pdl_wait();
  pdl_launch_dependents();

  const int MT = prm.MT, H = prm.H;
  const int NT = (int)ws.ctl[kCtlTokenTiles];
  // tensor memory: accumulators at columns 0 and 128, then the scale factors of the two h
  // buffers and of the two most recent weight tiles (natoms * 4 columns each)
  const uint32_t hsf_col = tmem + 256, wsf_col = tmem + 256 + 2 * natoms * 4;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int it = 0, hcount = 0;
      for (int j = blockIdx.x; j < NT && !abort_s; j += gridDim.x) {
        const int e = __ldg(&ws.tt_expert[j]);
        const int hb = hcount & 1, hn = hcount >> 1;
        if (hn > 0 && !mbar_wait(&h_empty[hb], (hn - 1) & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
          break;
        }
        unsigned char* hs = smem + hb * ustride;
        mbar_arrive_expect_tx(&h_full[hb], ubytes);
        for (int c = 0; c < nkc; ++c) tma_2d(hs + c * kTileBytes, &tm_h, c * 128, j * 128, &h_full[hb]);
        bulk_g2s(hs + nkc * kTileBytes, prm.sfb + (size_t)j * natoms * 512, natoms * 512,
                 &h_full[hb]);
        ++hcount;
        for (int mt = 0; mt < MT; ++mt) {
          const int s = it % nsw, n = it / nsw;
          if (n > 0 && !mbar_wait(&empty[s], (n - 1) & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
            break;
          }
          unsigned char* st = smem + 2 * ustride + kRhStaging + s * ustride;
          mbar_arrive_expect_tx(&full[s], ubytes);
          for (int c = 0; c < nkc; ++c)
            tma_2d(st + c * kTileBytes, &tm_w, c * 128, e * H + mt * 128, &full[s]);
          bulk_g2s(st + nkc * kTileBytes, prm.sfa + ((size_t)e * MT + mt) * natoms * 512,
                   natoms * 512, &full[s]);
          ++it;
        }
      }
      // no copy may still be in flight when the CTA exits
      const int used = it < nsw ? it : nsw;
      for (int i = 0; i < used; ++i) {
        const int c = it - 1 - i;
        (void)mbar_wait(&full[c % nsw], (c / nsw) & 1);
      }
      const int hused = hcount < 2 ? hcount : 2;
      for (int i = 0; i < hused; ++i) {
        const int c = hcount - 1 - i;
        (void)mbar_wait(&h_full[c & 1], (c >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int it = 0, hcount = 0, tcount = 0;
      for (int j = blockIdx.x; j < NT; j += gridDim.x) {
        // the previous h buffer is free once the MMAs issued so far have completed
        if (hcount > 0) commit(&h_empty[(hcount - 1) & 1]);
        const int hb = hcount & 1;
        if (!abort_s && !mbar_wait(&h_full[hb], (hcount >> 1) & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        fence_after();
        const uint32_t hsf0 = smem_u32(smem + hb * ustride + nkc * kTileBytes);
        for (int kb = 0; kb < natoms; ++kb)
          cp_sf(hsf_col + hb * natoms * 4 + 4 * kb, desc_sf(hsf0 + kb * 512));
        ++hcount;
        for (int mt = 0; mt < MT; ++mt, ++tcount) {
          const int buf = tcount & 1, use = tcount >> 1;
          if (use > 0 && !abort_s && !mbar_wait(&acc_empty[buf], (use - 1) & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
          }
          const int s = it % nsw, n = it / nsw;
          if (!abort_s && !mbar_wait(&full[s], n & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
          }
          fence_after();
          unsigned char* st = smem + 2 * ustride + kRhStaging + s * ustride;
          const uint32_t wsf = wsf_col + (tcount & 1) * natoms * 4;
          const uint32_t wsf0 = smem_u32(st + nkc * kTileBytes);
          for (int kb = 0; kb < natoms; ++kb) cp_sf(wsf + 4 * kb, desc_sf(wsf0 + kb * 512));
          const uint32_t h0 = smem_u32(smem + hb * ustride), w0 = smem_u32(st);
          const uint32_t hsf = hsf_col + hb * natoms * 4;
          for (int kb = 0; kb < natoms; ++kb) {
            const uint32_t off = (kb >> 2) * kTileBytes + (kb & 3) * 32;
            mma_nvf4(tmem + buf * kTileN, desc_sw128(h0 + off), desc_sw128(w0 + off), hsf + 4 * kb,
                     wsf + 4 * kb, kb > 0 ? 1u : 0u);
          }
          commit(&empty[s]);
          commit(&acc_full[buf]);
          ++it;
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..9)
    const int ew = warp - 2;
    const int quad = warp & 3;            // tensor-memory lanes 32*quad .. +31
    const int chalf = ew >> 2;            // columns 64*chalf .. +63
    const int col = quad * 32 + lane;     // accumulator row = slot of the token tile
    unsigned char* stg = smem + 2 * ustride + ew * (32 * 128);   // this warp's Y rows
    int tcount = 0;
    for (int j = blockIdx.x; j < NT; j += gridDim.x) {
      const int e = ws.tt_expert[j];
      const int slot0 = ws.tt_slot0[j], nval = ws.tt_n[j];
      for (int mt = 0; mt < MT; ++mt, ++tcount) {
        const int buf = tcount & 1, use = tcount >> 1;
        if (!abort_s && !mbar_wait(&acc_full[buf], use & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        __syncwarp();
        fence_after();
        const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16) + buf * kTileN + chalf * 64;
        uint32_t r0[32], r1[32];
        ld32(tbase, r0);
        ld32(tbase + 32, r1);
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        // this warp's slots quad*32 .. +31: nv of them are valid, the first nt go out by TMA
        const int nv = min(max(nval - quad * 32, 0), 32);
        const int nt = nv == 32 ? 32 : (nv & ~15);
        if (nv == 0) continue;
        if (nt > 0) {
          if (lane == 0) bulk_wait_read_all();   // the previous unit's store has read the rows
          __syncwarp();
        }
        // Y[slot][mt*128 + 64*chalf ..] = BF16(acc * md): 64 BF16 = 128 bytes of one slot row
        const float md = prm.mult[e * 3 + 2] * prm.dscale[e];
        uint4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i0 = (c * 8 + 2 * q) & 31;
            const uint32_t v0 = (c < 4) ? r0[i0] : r1[i0], v1 = (c < 4) ? r0[i0 + 1] : r1[i0 + 1];
            w[q] = (uint32_t)f32_to_bf16_rn(__uint_as_float(v0) * md) |
                   ((uint32_t)f32_to_bf16_rn(__uint_as_float(v1) * md) << 16);
          }
          v[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (lane < nt) {
          // row `lane` of the warp's box; 16-byte chunk c sits at c ^ (row & 7) (128-byte swizzle)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) = v[c];
        } else if (lane < nv) {
          uint4* dst = reinterpret_cast<uint4*>(ws.y + ((size_t)slot0 + col) * H + mt * 128 +
                                                chalf * 64);
#pragma unroll
          for (int c = 0; c < 8; ++c) dst[c] = v[c];
        }
        if (nt > 0) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(nt == 32 ? &tm_y32 : &tm_y16, stg, mt * 256 + chalf * 128,
                         slot0 + quad * 32);
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();   // the stores have completed before the CTA exits
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kRhTmemCols)
                 : "memory");
}

// ------------------------------------------------------------------ router GEMM (BF16)
// logits[T][E] = x[T][H] . Wr[E][H]^T on tcgen05.mma kind::f16 (BF16 x BF16 -> FP32 in tensor
// memory): A = 128 router rows, B = 128 tokens, K = 64 per stage (one 128-byte swizzle atom),
// four K = 16 instructions per stage. Warp 0: TMA producer; warp 1: MMA; warps 2..5: epilogue.
// Two CTAs per SM (3 stages of 32 KB and 256 tensor-memory columns each): one thread issues a
// CTA's 256 MMAs per tile, and a second CTA per SM is a second issuer.
constexpr int kRStages = 3;
constexpr int kRThreads = 192;
constexpr uint32_t kIdescBf16 = (1u << 4) | (1u << 7) | (1u << 10) |
                                ((uint32_t)(kTileN >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdescBf16), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(kRThreads, 2)
    k_tc_router(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                WsView ws) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t full[kRStages], empty[kRStages], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* smem = smem_raw + pad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = ws.T, H = ws.H, E = ws.E;
  if (tid == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    fence_mbar_init();
    abort_s = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_s)),
                 "r"(256)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_s;
  pdl_wait();
  pdl_launch_dependents();
  const int ME = (E + kTileM - 1) / kTileM, NTk = (T + kTileN - 1) / kTileN;
  const int ntiles = ME * NTk;
  const int nks = H / 64;
  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      for (int t = blockIdx.x; t < ntiles && !abort_s; t += gridDim.x) {
        const int me = t % ME, nt = t / ME;   // consecutive tiles share the token tile
        for (int ks = 0; ks < nks; ++ks, ++it) {
          const int s = it % kRStages, n = it / kRStages;
          if (n > 0 && !mbar_wait(&empty[s], (n - 1) & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
            break;
          }
          unsigned char* st = smem + s * 2 * kTileBytes;
          mbar_arrive_expect_tx(&full[s], 2 * kTileBytes);
          tma_2d(st, &tm_w, ks * 128, me * kTileM, &full[s]);
          tma_2d(st + kTileBytes, &tm_x, ks * 128, nt * kTileN, &full[s]);
        }
      }
      const int used = it < kRStages ? it : kRStages;
      for (int i = 0; i < used; ++i) {
        const int c = it - 1 - i;
        (void)mbar_wait(&full[c % kRStages], (c / kRStages) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0, tcount = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tcount) {
        const int buf = tcount & 1, use = tcount >> 1;
        if (use > 0 && !abort_s && !mbar_wait(&acc_empty[buf], (use - 1) & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        fence_after();
        for (int ks = 0; ks < nks; ++ks, ++it) {
          const int s = it % kRStages, n = it / kRStages;
          if (!abort_s && !mbar_wait(&full[s], n & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
          }
          fence_after();
          const uint32_t a0 = smem_u32(smem + s * 2 * kTileBytes);
          const uint32_t b0 = a0 + kTileBytes;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            mma_bf16(tmem + buf * kTileN, desc_sw128(a0 + q * 32), desc_sw128(b0 + q * 32),
                     (ks > 0 || q > 0) ? 1u : 0u);
          commit(&empty[s]);
        }
        commit(&acc_full[buf]);
      }
    }
  } else {
    const int quad = warp & 3;
    const int row = quad * 32 + lane;     // router row inside the tile
    int tcount = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tcount) {
      const int me = t % ME, nt = t / ME;
      const int buf = tcount & 1, use = tcount >> 1;
      if (!abort_s && !mbar_wait(&acc_full[buf], use & 1)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
      }
      __syncwarp();
      fence_after();
      const int e = me * kTileM + row;
      const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16) + buf * kTileN;
      for (int c0 = 0; c0 < kTileN; c0 += 32) {
        uint32_t r[32];
        ld32(tbase + c0, r);
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int tok = nt * kTileN + c0 + q;
          if (tok < T && e < E) ws.logits[(size_t)tok * E + e] = __uint_as_float(r[q]);
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256)
                 : "memory");
}

// ------------------------------------------------------------------ activations by pslot
// W4A4 activations of the grouped path in one pass: 64 threads per token quantise its row
// (four 16-element blocks per thread, the quantiser Q with the gate/up input scale), publish the
// codes and scales by token, and write the token's k copies into the padded permuted operand
// ("pslot" = 128 * token tile + rank in the tile) with their scale-factor atom words.
constexpr int kXqTok = 4;   // tokens per CTA

__global__ void __launch_bounds__(64 * kXqTok) k_xquant_perm(const uint16_t* __restrict__ x,
                                                             WsView ws, float xS, float x_inv6S) {
  __shared__ int pslot_s[kXqTok][32];
  const int H = ws.H, k = ws.k;
  const int tl = threadIdx.x >> 6, q = threadIdx.x & 63;
  const int t = blockIdx.x * kXqTok + tl;
  pdl_wait();
  pdl_launch_dependents();
  if (t < ws.T && q < k) {
    const int s = ws.slot_of[(size_t)t * k + q], e = ws.idx[(size_t)t * k + q];
    pslot_s[tl][q] = ws.ttbase[e] * 128 + (s - ws.offsets[e]);
  }
  __syncthreads();
  if (t >= ws.T) return;
  // every lane of a warp runs each round (the shuffles below need all 32), whether or not its
  // group g lies inside the row
  for (int gb = 0; gb < H / 64; gb += 64) {
    const int g = gb + q;
    const bool act = g < H / 64;
    uint32_t cw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u}, sfw = 0;
    if (act) {
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H + (size_t)g * 64);
      uint4 u[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = src[i];
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        const uint32_t w8[8] = {u[2 * blk].x, u[2 * blk].y, u[2 * blk].z, u[2 * blk].w,
                                u[2 * blk + 1].x, u[2 * blk + 1].y, u[2 * blk + 1].z,
                                u[2 * blk + 1].w};
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[2 * i] = bf16_lo(w8[i]);
          v[2 * i + 1] = bf16_hi(w8[i]);
        }
        uint32_t c2[2];
        const uint32_t sf = quantize16(v, xS, x_inv6S, c2);
        cw[2 * blk] = c2[0];
        cw[2 * blk + 1] = c2[1];
        sfw |= sf << (8 * blk);
      }
    }
    // Lane l holds the 32 code bytes of group g; one warp covers 1 KB of the row. Two shuffle
    // rounds give lane l the 16-byte chunks l and 32 + l of that 1 KB (groups gw + l/2 and
    // gw + 16 + l/2), so every store below writes up to 512 contiguous bytes per warp.
    const int lane = threadIdx.x & 31;
    const int gw = gb + (q & ~31);           // first group of this warp
    uint32_t ca[4], cb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo_a = __shfl_sync(0xFFFFFFFFu, cw[i], lane >> 1);
      const uint32_t hi_a = __shfl_sync(0xFFFFFFFFu, cw[4 + i], lane >> 1);
      const uint32_t lo_b = __shfl_sync(0xFFFFFFFFu, cw[i], 16 + (lane >> 1));
      const uint32_t hi_b = __shfl_sync(0xFFFFFFFFu, cw[4 + i], 16 + (lane >> 1));
      ca[i] = (lane & 1) ? hi_a : lo_a;
      cb[i] = (lane & 1) ? hi_b : lo_b;
    }
    const bool okA = gw + (lane >> 1) < H / 64, okB = gw + 16 + (lane >> 1) < H / 64;
    const uint4 va = make_uint4(ca[0], ca[1], ca[2], ca[3]);
    const uint4 vb = make_uint4(cb[0], cb[1], cb[2], cb[3]);
    const size_t wofs = (size_t)gw * 32;     // byte offset of this warp's 1 KB in a row
    uint4* xd = reinterpret_cast<uint4*>(ws.xq + (size_t)t * (H / 2) + wofs);
    if (okA) xd[lane] = va;
    if (okB) xd[32 + lane] = vb;
    if (act) *reinterpret_cast<uint32_t*>(ws.xsf + (size_t)t * (H / 16) + (size_t)g * 4) = sfw;
    for (int j = 0; j < k; ++j) {
      uint4* pd = reinterpret_cast<uint4*>(ws.xq_perm + (size_t)pslot_s[tl][j] * (H / 2) + wofs);
      if (okA) pd[lane] = va;
      if (okB) pd[32 + lane] = vb;
    }
  }
}

// Scale-factor atoms of the permuted activations, from the token-order scales: warp (token tile
// j, 4 groups of 64 elements) writes the 512-byte atom of each group with one 16-byte store per
// lane; lane l's 16 bytes are the 4 scales of rows l, l + 32, l + 64, l + 96 of the tile.
__global__ void __launch_bounds__(256) k_xsf_atoms(WsView ws) {
  const int G = ws.H / 64;                     // atoms per tile row (a multiple of 4)
  const int lane = threadIdx.x & 31;
  const int wid = blockIdx.x * 8 + (threadIdx.x >> 5);
  pdl_wait();
  pdl_launch_dependents();
  const int NT = (int)ws.ctl[kCtlTokenTiles];
  const int j = wid / (G / 4), g0 = (wid % (G / 4)) * 4;
  if (j >= NT) return;
  const int slot0 = ws.tt_slot0[j], nval = ws.tt_n[j];
  int tok[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = lane + 32 * i;
    tok[i] = r < nval ? ws.perm[slot0 + r] : -1;
  }
  // the 4 groups' scale words of a row are 16 contiguous bytes of the token-order scales
  uint4 sv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    sv[i] = tok[i] >= 0 ? *reinterpret_cast<const uint4*>(ws.xsf + (size_t)tok[i] * (G * 4) + g0 * 4)
                        : make_uint4(0u, 0u, 0u, 0u);
  unsigned char* dst = ws.xsf_atoms + ((size_t)j * G + g0) * 512 + lane * 16;
  *reinterpret_cast<uint4*>(dst) = make_uint4(sv[0].x, sv[1].x, sv[2].x, sv[3].x);
  *reinterpret_cast<uint4*>(dst + 512) = make_uint4(sv[0].y, sv[1].y, sv[2].y, sv[3].y);
  *reinterpret_cast<uint4*>(dst + 1024) = make_uint4(sv[0].z, sv[1].z, sv[2].z, sv[3].z);
  *reinterpret_cast<uint4*>(dst + 1536) = make_uint4(sv[0].w, sv[1].w, sv[2].w, sv[3].w);
}

// ------------------------------------------------------------------ W4A16 grouped experts
// Tensor cores need both operands in one 16-bit type, and NVFP4 x BF16 has no MMA kind, so the
// W4A16 grouped path runs tcgen05 kind::f16 on f16 operands that hold the values exactly:
//   A (weights): E2M1 code x E4M3 scale (<= 6 significant bits, |v| <= 2688: exact in f16),
//     dequantised in shared memory by converter warps from the TMA-staged FP4 codes;
//   B (activations): x * 2^-s per token (gate/up) and BF16 h * 2^-s per slot (down), with s
//     putting the row's max |value| in [2^14, 2^15) (exact, as in the narrow-call path);
// the epilogues restore 2^s. K = 64 per stage. Gate/up: one 128 x 256 MMA per K = 16 step, the
// 128 slots of a token tile as M and the 128 gate and 128 up rows of an intermediate tile as N,
// interleaved by 16 (rows 32b .. 32b+15 gate, +16 .. +31 up), so that one epilogue thread holds
// a slot's gate and up values of a 16-element block of h side by side. Down: 128 weight rows x
// 128 slots (or the resident-h kernel k_tc16_dn below).
constexpr int kT16Stages = 6;   // load stages (activation tile, FP4 codes, scale atoms)
constexpr int kT16Conv = 2;     // dequantised weight buffers
constexpr int kT16Threads = 10 * 32;   // producer, MMA, 4 converter warps, 4 epilogue warps
constexpr uint32_t kIdescF16 = (1u << 4) | ((uint32_t)(kTileN >> 3) << 17) |
                               ((uint32_t)(kTileM >> 4) << 24);   // f16 x f16 -> f32, 128x128

// f16 x f16 -> f32, 128 x 256 (gate/up: 128 slots x 256 weight rows)
constexpr uint32_t kIdescF16N256 = (1u << 4) | ((uint32_t)(256 >> 3) << 17) |
                                   ((uint32_t)(kTileM >> 4) << 24);

__device__ __forceinline__ void mma_f16_n256(uint32_t d, uint64_t a, uint64_t b,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdescF16N256), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdescF16), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void t16_epi_sync() {  // the 4 epilogue warps
  asm volatile("bar.sync 3, 128;" ::: "memory");
}

// Shared memory (bytes): kT16Stages load stages, each B (16 KB, SW128), the raw FP4 codes
// (gate/up: 2 x 128 rows x 32 B) and the scale-factor atoms (gate/up 2, down 1); then kT16Conv
// buffers of dequantised A (f16, SW128; gate/up: gate 16 KB + up 16 KB). The load ring and the
// dequantised buffers are separate rings: a load stage is refilled once its MMAs have run,
// without waiting for a conversion slot, so six stages of copies stay in flight while two
// buffers alternate between the converters and the MMAs.
template <bool DOWN>
struct T16 {
  static constexpr int kConv = DOWN ? 16384 : 32768;
  static constexpr int kB = 16384;
  static constexpr int kRaw = DOWN ? 4096 : 8192;
  static constexpr int kSf = DOWN ? 512 : 1024;
  static constexpr int kStage = ((kB + kRaw + kSf) + 1023) / 1024 * 1024;
  static constexpr int kTmemCols = DOWN ? 256 : 512;
  static constexpr int kYStage = kTileN * kYStride * 2;   // down: transposed BF16 Y tile
  static constexpr int kSmem =
      kT16Stages * kStage + kT16Conv * kConv + (DOWN ? kYStage : 0) + 512 + 1024;
};
static_assert(T16<false>::kSmem <= 232448 && T16<true>::kSmem <= 232448, "k_tc16 shared memory");

template <bool DOWN>
__global__ void __launch_bounds__(kT16Threads, 1)
    k_tc16(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
           const __grid_constant__ CUtensorMap tm_b, TcParams prm, WsView ws) {
  using L = T16<DOWN>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t full[kT16Stages], empty[kT16Stages];
  __shared__ uint64_t conv_full[kT16Conv], conv_empty[kT16Conv];
  __shared__ uint64_t acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* smem = smem_raw + pad;
  unsigned char* convb = smem + kT16Stages * L::kStage;             // dequantised A buffers
  unsigned char* ystage = convb + kT16Conv * L::kConv;              // down: Y tile
  float* colfac = reinterpret_cast<float*>(ystage + (DOWN ? L::kYStage : 0));   // [128]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kT16Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int c = 0; c < kT16Conv; ++c) {
      mbar_init(&conv_full[c], 4);
      mbar_init(&conv_empty[c], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    fence_mbar_init();
    abort_s = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_s)),
                 "r"(L::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_s;
  pdl_wait();
  pdl_launch_dependents();

  const int NT = (int)ws.ctl[kCtlTokenTiles];
  const int ntiles = NT * prm.MT;
  const int H = prm.H, I = prm.I;
  const int nks = DOWN ? I / 64 : H / 64;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int it = 0;
      for (int t = blockIdx.x; t < ntiles && !abort_s; t += gridDim.x) {
        const int j = t / prm.MT, mt = t % prm.MT;
        const int e = __ldg(&ws.tt_expert[j]);
        for (int ks = 0; ks < nks; ++ks, ++it) {
          const int s = it % kT16Stages, n = it / kT16Stages;
          if (n > 0 && !mbar_wait(&empty[s], (n - 1) & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
            break;
          }
          unsigned char* st = smem + s * L::kStage;
          unsigned char* bt = st;
          unsigned char* raw = bt + L::kB;
          unsigned char* sf = raw + L::kRaw;
          mbar_arrive_expect_tx(&full[s], L::kB + L::kRaw + L::kSf);
          if (!DOWN) {
            tma_2d(raw, &tm_a0, ks * 32, e * I + mt * 128, &full[s]);
            tma_2d(raw + 4096, &tm_a1, ks * 32, e * I + mt * 128, &full[s]);
            // scale atoms of the two 64-index intermediate tiles (each: gate and up rows
            // interleaved by 16)
            for (int h2 = 0; h2 < 2; ++h2)
              bulk_g2s(sf + h2 * 512,
                       prm.sfa + (((size_t)e * (I / 64) + 2 * mt + h2) * (H / 64) + ks) * 512, 512,
                       &full[s]);
          } else {
            tma_2d(raw, &tm_a0, ks * 32, e * H + mt * 128, &full[s]);
            bulk_g2s(sf, prm.sfa + (((size_t)e * (H / 128) + mt) * (I / 64) + ks) * 512, 512,
                     &full[s]);
          }
          tma_2d(bt, &tm_b, ks * 128, j * 128, &full[s]);
        }
      }
      const int used = it < kT16Stages ? it : kT16Stages;
      for (int i = 0; i < used; ++i) {
        const int c = it - 1 - i;
        (void)mbar_wait(&full[c % kT16Stages], (c / kT16Stages) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int it = 0, tcount = 0;
      const uint32_t bufcols = DOWN ? kTileN : 2 * kTileN;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tcount) {
        const int buf = tcount & 1, use = tcount >> 1;
        if (use > 0 && !abort_s && !mbar_wait(&acc_empty[buf], (use - 1) & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        fence_after();
        const uint32_t d0 = tmem + buf * bufcols;
        for (int ks = 0; ks < nks; ++ks, ++it) {
          // load stage s holds B; buffer c holds the dequantised A (its converters waited for
          // stage s to land before they signalled c)
          const int s = it % kT16Stages, c = it % kT16Conv;
          if (!abort_s && !mbar_wait(&conv_full[c], (it / kT16Conv) & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
          }
          fence_after();
          const uint32_t a0 = smem_u32(convb + c * L::kConv), b0 = smem_u32(smem + s * L::kStage);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t acc = (ks > 0 || q > 0) ? 1u : 0u;
            if (DOWN)
              mma_f16(d0, desc_sw128(a0 + q * 32), desc_sw128(b0 + q * 32), acc);
            else   // M = the 128 slots, N = the 256 gate/up weight rows
              mma_f16_n256(d0, desc_sw128(b0 + q * 32), desc_sw128(a0 + q * 32), acc);
          }
          commit(&empty[s]);
          commit(&conv_empty[c]);
        }
        commit(&acc_full[buf]);
      }
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------------- converters (warps 2..5)
    // thread ct owns A row ct (gate/up: gate row ct and up row ct) of every stage
    const int ct = tid - 64;
    int it = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      for (int ks = 0; ks < nks; ++ks, ++it) {
        const int s = it % kT16Stages, n = it / kT16Stages;
        const int cb = it % kT16Conv, cu = it / kT16Conv;
        if (!abort_s && !mbar_wait(&full[s], n & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        // buffer cb is free once the MMAs of its previous use have run
        if (cu > 0 && !abort_s && !mbar_wait(&conv_empty[cb], (cu - 1) & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        const unsigned char* raw = smem + s * L::kStage + L::kB;
        const unsigned char* sf = raw + L::kRaw;
        unsigned char* st = convb + cb * L::kConv;
#pragma unroll
        for (int mat = 0; mat < (DOWN ? 1 : 2); ++mat) {
          const uint4* src = reinterpret_cast<const uint4*>(raw + mat * 4096 + ct * 32);
          const uint4 c0 = src[0], c1 = src[1];
          // the row's 4 scale bytes (blocks of 16 along this stage's 64 K)
          // atom rows: gate and up rows of a 64-index tile interleaved by 16
          const int rr = DOWN ? ct : ((ct & 63) >> 4) * 32 + mat * 16 + (ct & 15);
          const unsigned char* atom = sf + (DOWN ? 0 : (ct >> 6) * 512);
          const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(atom + (rr & 31) * 16 + (rr >> 5) * 4);
          const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          // gate/up: row ct of matrix mat is row rb of the 256-row weight tile, the gate and up
          // rows of each 16-index block side by side (rows 32b .. 32b+15 gate, +16 .. +31 up)
          const int rb = DOWN ? ct : ((ct >> 4) * 32 + mat * 16 + (ct & 15));
          unsigned char* row = st + (rb >> 3) * 1024 + (rb & 7) * 128;
          const uint32_t s01 = e4m3x2_to_f16x2(sc4), s23 = e4m3x2_to_f16x2(sc4 >> 16);
#pragma unroll
          for (int c = 0; c < 8; ++c) {   // chunk c: elements 8c .. 8c+7 = code word c
            const uint32_t sp = (c < 4) ? s01 : s23;
            uint32_t f[4];
            e2m1x8_to_f16x2x4(w[c], f);
            uint4 o;
            if (c & 2) {   // blocks 1 and 3 of the stage: the high half of the pair
              o = make_uint4(hmul2_hi(f[0], sp), hmul2_hi(f[1], sp), hmul2_hi(f[2], sp),
                             hmul2_hi(f[3], sp));
            } else {
              o = make_uint4(hmul2_lo(f[0], sp), hmul2_lo(f[1], sp), hmul2_lo(f[2], sp),
                             hmul2_lo(f[3], sp));
            }
            *reinterpret_cast<uint4*>(row + ((c ^ (ct & 7)) << 4)) = o;
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&conv_full[cb]);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 6..9)
    const int et = tid - 192;               // 0..127
    const int quad = warp & 3;              // tensor-memory lanes 32*quad .. +31
    const int row = quad * 32 + lane;       // accumulator row of this thread
    int tcount = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tcount) {
      const int j = t / prm.MT, mt = t % prm.MT;
      const int buf = tcount & 1, use = tcount >> 1;
      const int e = ws.tt_expert[j];
      const int slot0 = ws.tt_slot0[j], nval = ws.tt_n[j];
      if (DOWN) {
        // per column (slot) factor 2^s of the slot's h, or fl32(6 S_down) in W4A8
        float f = 0.0f;
        if (et < nval)
          f = prm.a8 ? __fmul_rn(6.0f, prm.dscale[e])
                     : __int_as_float((127 + amax_shift(__uint_as_float(ws.slot_amax[slot0 + et])))
                                      << 23);
        colfac[et] = f;
        t16_epi_sync();
      }
      if (!abort_s && !mbar_wait(&acc_full[buf], use & 1)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
      }
      __syncwarp();
      fence_after();
      if (!DOWN) {
        // accumulator row = slot `row` of the token tile; columns 32b .. 32b+15 are the gate and
        // 32b+16 .. 32b+31 the up products of intermediate indices mt*128 + 16b .. +15: one
        // tensor-memory load per 16-element block of h, SiLU*up in registers, 32 (BF16) or 16
        // (E4M3) contiguous bytes of the slot's h row per block
        const uint32_t tb = tmem + ((uint32_t)(quad * 32) << 16) + buf * (2 * kTileN);
        const float mg = prm.mult[e * 3 + 0], mu = prm.mult[e * 3 + 1];
        const bool valid = row < nval;
        const float fx = valid ? ws.xfac[ws.perm[slot0 + row]] : 0.0f;
        const size_t hrow = (size_t)(slot0 + (valid ? row : 0)) * I + mt * 128;
        float amax = 0.0f;
        for (int blk = 0; blk < 8; ++blk) {
          uint32_t r[32];
          ld32(tb + blk * 32, r);
          if (blk == 7) {   // every column is in registers: the buffer goes back to the MMA warp
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
          }
          float h[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float gv = __uint_as_float(r[i]) * mg * fx;
            const float uv = __uint_as_float(r[16 + i]) * mu * fx;
            h[i] = (gv / (1.0f + expf(-gv))) * uv;
          }
          if (!valid) continue;
          if (prm.a8) {
            // W4A8: h -> E4M3 with the down matrix's scale (dinv6 = fl32(1/fl32(6 S_down)))
            const float r8 = prm.dinv6[e];
            uint32_t cw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int i = 0; i < 16; ++i) cw[i >> 2] |= a8_encode(h[i], r8) << (8 * (i & 3));
            *reinterpret_cast<uint4*>(ws.hq + hrow + blk * 16) =
                make_uint4(cw[0], cw[1], cw[2], cw[3]);
          } else {
            uint32_t hw[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t lo = f32_to_bf16_rn(h[2 * i]), hi = f32_to_bf16_rn(h[2 * i + 1]);
              hw[i] = lo | (hi << 16);
              // |h| of the BF16 values, for the down operand's per-slot scaling
              amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(lo << 16)),
                                       fabsf(__uint_as_float(hi << 16))));
            }
            uint4* dst = reinterpret_cast<uint4*>(ws.h16 + hrow + blk * 16);
            dst[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            dst[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
          }
        }
        if (valid && !prm.a8) atomicMax(&ws.slot_amax[slot0 + row], __float_as_uint(amax));
      } else {
        const uint32_t tb = tmem + ((uint32_t)(quad * 32) << 16) + buf * kTileN;
        const float md = prm.mult[e * 3 + 2];
        uint16_t* yt = reinterpret_cast<uint16_t*>(ystage);
        for (int c0 = 0; c0 < kTileN; c0 += 32) {
          uint32_t r[32];
          ld32(tb + c0, r);
#pragma unroll
          for (int q = 0; q < 32; ++q)
            yt[(c0 + q) * kYStride + row] =
                f32_to_bf16_rn(__uint_as_float(r[q]) * md * colfac[c0 + q]);
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        t16_epi_sync();
        for (int id = et; id < kTileN * (kTileM / 8); id += 128) {
          const int col = id >> 4, r8 = id & 15;
          if (col < nval)
            *reinterpret_cast<uint4*>(ws.y + (size_t)(slot0 + col) * H + mt * 128 + r8 * 8) =
                *reinterpret_cast<const uint4*>(yt + col * kYStride + r8 * 8);
        }
      }
      if (DOWN) t16_epi_sync();   // colfac and the Y tile are reused by the next tile
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(L::kTmemCols)
                 : "memory");
}

// W4A16 down GEMM with the operands' roles swapped: A = the h tile of one 128-slot token tile
// (f16, all I columns, resident in shared memory while the CTA runs every 256-row weight tile of
// that token tile), B = 256 dequantised down-weight rows x 64 K per stage, D = [slot][row]
// (M = 128, N = 256) in tensor memory. The h tile is staged once per token tile instead of once
// per weight tile. Each epilogue thread owns one slot; per 64 columns an epilogue warp writes its
// 32 slots' Y rows into a 128-byte swizzled staging box and stores the box with TMA (plain row
// stores for a ragged tile's last rows, or for every row when the h tile leaves no room for the
// staging). As in k_tc16, the ring of TMA load stages (codes and scale atoms) is separate from
// the two dequantised-weight buffers.
constexpr int kDnN = 256;
constexpr uint32_t kIdescDn = (1u << 4) | ((uint32_t)(kDnN >> 3) << 17) |
                              ((uint32_t)(kTileM >> 4) << 24);   // f16 x f16 -> f32, 128x256
constexpr int kDnConv = kDnN * 128;                 // 256 rows x 128 B (64 f16), SW128
constexpr int kDnRaw = kDnN * 32;                   // 256 rows x 64 FP4 codes
constexpr int kDnSf = 2 * 512;                      // two 128-row scale-factor atoms
constexpr int kDnLStage = kDnRaw + kDnSf;          // 9 KB load stage, a multiple of 1 KB
constexpr int kDnConvBufs = 2;                      // dequantised B buffers
constexpr int kDnYStaging = 4 * 2 * 4096;           // per epilogue warp: two 32-row x 128 B Y boxes
constexpr int kDnMaxStages = 8;

__device__ __forceinline__ void mma_f16_dn(uint32_t d, uint64_t a, uint64_t b,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdescDn), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(kT16Threads, 1)
    k_tc16_dn(const __grid_constant__ CUtensorMap tm_raw, const __grid_constant__ CUtensorMap tm_h,
              const __grid_constant__ CUtensorMap tm_y32, const __grid_constant__ CUtensorMap tm_y16,
              TcParams prm, WsView ws, int nst, int ybox) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t full[kDnMaxStages], empty[kDnMaxStages];
  __shared__ uint64_t conv_full[kDnConvBufs], conv_empty[kDnConvBufs];
  __shared__ uint64_t acc_full[2], acc_empty[2], a_full, a_empty;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* smem = smem_raw + pad;
  const int H = prm.H, I = prm.I;
  const int nks = I / 64;
  // the h tile, two dequantised weight buffers, then the ring of load stages (FP4 codes and
  // scale atoms): a load stage is refilled once its buffer's MMAs have run, without waiting for
  // a conversion slot, so nst stages of copies stay in flight
  unsigned char* atile = smem;                                   // [nks][128 rows x 128 B]
  unsigned char* convb = smem + (size_t)nks * 16384;             // [2][256 rows x 128 B]
  unsigned char* stages = convb + kDnConvBufs * kDnConv;
  unsigned char* ystg = stages + (size_t)nst * kDnLStage;       // [4 warps][2][32 rows x 128 B]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int c = 0; c < kDnConvBufs; ++c) {
      mbar_init(&conv_full[c], 4);
      mbar_init(&conv_empty[c], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(&a_full, 1);
    mbar_init(&a_empty, 1);
    fence_mbar_init();
    abort_s = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_s)),
                 "r"(2 * kDnN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_s;
  pdl_wait();
  pdl_launch_dependents();

  // units (token tile j, 256-row weight tile nt), a contiguous share per CTA so that consecutive
  // units reuse the staged h tile
  const int nts = H / kDnN;
  const int nunits = (int)ws.ctl[kCtlTokenTiles] * nts;
  const int u0 = (int)(((long long)nunits * blockIdx.x) / gridDim.x);
  const int u1 = (int)(((long long)nunits * (blockIdx.x + 1)) / gridDim.x);

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int it = 0, jprev = -1, jcount = 0;
      for (int u = u0; u < u1 && !abort_s; ++u) {
        const int j = u / nts, nt = u % nts;
        const int e = __ldg(&ws.tt_expert[j]);
        if (j != jprev) {
          if (jcount > 0 && !mbar_wait(&a_empty, (jcount - 1) & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
            break;
          }
          mbar_arrive_expect_tx(&a_full, (uint32_t)nks * 16384u);
          for (int ks = 0; ks < nks; ++ks) tma_2d(atile + ks * 16384, &tm_h, ks * 128, j * 128, &a_full);
          jprev = j;
          ++jcount;
        }
        for (int ks = 0; ks < nks; ++ks, ++it) {
          const int s = it % nst, n = it / nst;
          if (n > 0 && !mbar_wait(&empty[s], (n - 1) & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
            break;
          }
          unsigned char* raw = stages + (size_t)s * kDnLStage;
          unsigned char* sf = raw + kDnRaw;
          mbar_arrive_expect_tx(&full[s], kDnRaw + kDnSf);
          tma_2d(raw, &tm_raw, ks * 32, e * H + nt * kDnN, &full[s]);
          tma_2d(raw + 4096, &tm_raw, ks * 32, e * H + nt * kDnN + 128, &full[s]);
          for (int h2 = 0; h2 < 2; ++h2)
            bulk_g2s(sf + h2 * 512,
                     prm.sfa + (((size_t)e * (H / 128) + 2 * nt + h2) * (I / 64) + ks) * 512, 512,
                     &full[s]);
        }
      }
      const int used = it < nst ? it : nst;
      for (int i = 0; i < used; ++i) {
        const int c = it - 1 - i;
        (void)mbar_wait(&full[c % nst], (c / nst) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int it = 0, tcount = 0, jprev = -1, jcount = 0;
      for (int u = u0; u < u1; ++u, ++tcount) {
        const int j = u / nts;
        if (j != jprev) {
          if (!abort_s && !mbar_wait(&a_full, jcount & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
          }
          jprev = j;
          ++jcount;
        }
        const int buf = tcount & 1, use = tcount >> 1;
        if (use > 0 && !abort_s && !mbar_wait(&acc_empty[buf], (use - 1) & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        fence_after();
        const uint32_t d0 = tmem + buf * kDnN;
        for (int ks = 0; ks < nks; ++ks, ++it) {
          const int s = it % nst, c = it % kDnConvBufs;
          if (!abort_s && !mbar_wait(&conv_full[c], (it / kDnConvBufs) & 1)) {
            record_status(ws.ctl, kStTimeout);
            abort_s = 1;
          }
          fence_after();
          const uint32_t a0 = smem_u32(atile + ks * 16384);
          const uint32_t b0 = smem_u32(convb + c * kDnConv);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            mma_f16_dn(d0, desc_sw128(a0 + q * 32), desc_sw128(b0 + q * 32),
                       (ks > 0 || q > 0) ? 1u : 0u);
          commit(&empty[s]);
          commit(&conv_empty[c]);
        }
        commit(&acc_full[buf]);
        // the h tile may be replaced once this token tile's last MMA has read it
        if (u + 1 == u1 || (u + 1) / nts != j) commit(&a_empty);
      }
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------------- converters (warps 2..5)
    // thread ct owns B rows ct and ct + 128 of every stage
    const int ct = tid - 64;
    int it = 0;
    for (int u = u0; u < u1; ++u) {
      for (int ks = 0; ks < nks; ++ks, ++it) {
        const int s = it % nst, n = it / nst;
        const int cb = it % kDnConvBufs, cu = it / kDnConvBufs;
        if (!abort_s && !mbar_wait(&full[s], n & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        // buffer cb is free once the MMAs of its previous use have run
        if (cu > 0 && !abort_s && !mbar_wait(&conv_empty[cb], (cu - 1) & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        unsigned char* st = convb + cb * kDnConv;
        const unsigned char* raw = stages + (size_t)s * kDnLStage;
        const unsigned char* sf = raw + kDnRaw;
#pragma unroll
        for (int mat = 0; mat < 2; ++mat) {
          const uint4* src = reinterpret_cast<const uint4*>(raw + mat * 4096 + ct * 32);
          const uint4 c0 = src[0], c1 = src[1];
          // the row's 4 scale bytes (blocks of 16 along this stage's 64 K)
          const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(sf + mat * 512 + (ct & 31) * 16 +
                                                                  (ct >> 5) * 4);
          const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          unsigned char* row = st + mat * 16384 + (ct >> 3) * 1024 + (ct & 7) * 128;
          const uint32_t s01 = e4m3x2_to_f16x2(sc4), s23 = e4m3x2_to_f16x2(sc4 >> 16);
#pragma unroll
          for (int c = 0; c < 8; ++c) {   // chunk c: elements 8c .. 8c+7 = code word c
            const uint32_t sp = (c < 4) ? s01 : s23;
            uint32_t f[4];
            e2m1x8_to_f16x2x4(w[c], f);
            uint4 o;
            if (c & 2) {
              o = make_uint4(hmul2_hi(f[0], sp), hmul2_hi(f[1], sp), hmul2_hi(f[2], sp),
                             hmul2_hi(f[3], sp));
            } else {
              o = make_uint4(hmul2_lo(f[0], sp), hmul2_lo(f[1], sp), hmul2_lo(f[2], sp),
                             hmul2_lo(f[3], sp));
            }
            *reinterpret_cast<uint4*>(row + ((c ^ (ct & 7)) << 4)) = o;
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&conv_full[cb]);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 6..9)
    const int quad = warp & 3;              // tensor-memory lanes 32*quad .. +31
    const int row = quad * 32 + lane;       // slot of the token tile
    unsigned char* stg = ystg + (warp - 6) * 8192;   // this warp's two Y boxes
    int tcount = 0, ycount = 0;
    for (int u = u0; u < u1; ++u, ++tcount) {
      const int j = u / nts, nt = u % nts;
      const int buf = tcount & 1, use = tcount >> 1;
      const int e = ws.tt_expert[j];
      const int slot0 = ws.tt_slot0[j], nval = ws.tt_n[j];
      // Y = BF16(acc * md * 2^s of the slot), or * fl32(6 S_down) in W4A8
      float f = 0.0f;
      if (row < nval)
        f = prm.mult[e * 3 + 2] *
            (prm.a8 ? __fmul_rn(6.0f, prm.dscale[e])
                    : __int_as_float((127 + amax_shift(__uint_as_float(ws.slot_amax[slot0 + row])))
                                     << 23));
      if (!abort_s && !mbar_wait(&acc_full[buf], use & 1)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
      }
      __syncwarp();
      fence_after();
      const uint32_t tb = tmem + ((uint32_t)(quad * 32) << 16) + buf * kDnN;
      // this warp's slots quad*32 .. +31: nv of them are valid, the first ntm go out by TMA
      // (32- or 16-row boxes of 64 BF16 = 128 bytes per row, staged 128-byte swizzled), the
      // rest of a ragged tile as plain row stores (all of them when the staging did not fit:
      // ybox = 0)
      const int nv = min(max(nval - quad * 32, 0), 32);
      const int ntm = !ybox ? 0 : nv == 32 ? 32 : (nv & ~15);
      for (int c0 = 0; c0 < kDnN; c0 += 64, ++ycount) {
        uint32_t r0[32], r1[32];
        ld32(tb + c0, r0);
        ld32(tb + c0 + 32, r1);
        if (c0 + 64 == kDnN) {   // every column is in registers: the buffer goes back
          fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
        if (nv == 0) continue;
        uint4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i0 = (c * 8 + 2 * q) & 31;
            const uint32_t v0 = (c < 4) ? r0[i0] : r1[i0], v1 = (c < 4) ? r0[i0 + 1] : r1[i0 + 1];
            w[q] = (uint32_t)f32_to_bf16_rn(__uint_as_float(v0) * f) |
                   ((uint32_t)f32_to_bf16_rn(__uint_as_float(v1) * f) << 16);
          }
          v[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        unsigned char* sb = stg + (ycount & 1) * 4096;
        if (ntm > 0) {
          if (lane == 0) bulk_wait_read_but1();   // the store that last used sb has read it
          __syncwarp();
        }
        if (lane < ntm) {
          // row `lane` of the box; 16-byte chunk c sits at c ^ (row & 7) (128-byte swizzle)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(sb + lane * 128 + ((c ^ (lane & 7)) << 4)) = v[c];
        } else if (lane < nv) {
          uint4* dst =
              reinterpret_cast<uint4*>(ws.y + (size_t)(slot0 + row) * H + nt * kDnN + c0);
#pragma unroll
          for (int c = 0; c < 8; ++c) dst[c] = v[c];
        }
        if (ntm > 0) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(ntm == 32 ? &tm_y32 : &tm_y16, sb, (nt * kDnN + c0) * 2,
                         slot0 + quad * 32);
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();   // the stores have completed before the CTA exits
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(2 * kDnN)
                 : "memory");
}

// W4A16 activations by padded slot: 64 threads per token find the token's max |x|, then write
// f16(x * 2^-s) into each of its k slots' rows and 2^s to xfac (exact; see above).
__global__ void __launch_bounds__(64 * kXqTok) k_xprep16_perm(const uint16_t* __restrict__ x,
                                                              WsView ws, int a8, float xS,
                                                              float r8) {
  __shared__ int pslot_s[kXqTok][32];
  __shared__ float am_s[kXqTok][2];
  const int H = ws.H, k = ws.k;
  const int tl = threadIdx.x >> 6, q = threadIdx.x & 63, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kXqTok + tl;
  pdl_wait();
  pdl_launch_dependents();
  const bool live = t < ws.T;
  if (live && q < k) {
    const int s = ws.slot_of[(size_t)t * k + q], e = ws.idx[(size_t)t * k + q];
    pslot_s[tl][q] = ws.ttbase[e] * 128 + (s - ws.offsets[e]);
  }
  float m = 0.0f;
  if (live)
    for (int g = q; g < H / 8; g += 64) {
      const uint4 u = reinterpret_cast<const uint4*>(x + (size_t)t * H)[g];
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w4[i])), fabsf(bf16_hi(w4[i]))));
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if (lane == 0) am_s[tl][q >> 5] = m;
  __syncthreads();
  if (!live) return;
  if (a8) {
    // W4A8: the E4M3 code of every element (published in token order) and its value as the f16
    // operand (exact); the scale fl32(6 S) goes to xfac
    if (q == 0) ws.xfac[t] = __fmul_rn(6.0f, xS);
    for (int g = q; g < H / 8; g += 64) {
      const uint4 u = reinterpret_cast<const uint4*>(x + (size_t)t * H)[g];
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
      uint32_t cw[2] = {0u, 0u}, o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        cw[i >> 1] |= (a8_encode(bf16_lo(w4[i]), r8) | (a8_encode(bf16_hi(w4[i]), r8) << 8))
                      << (16 * (i & 1));
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = e4m3x2_to_f16x2(cw[i >> 1] >> (16 * (i & 1)));
      *reinterpret_cast<uint2*>(ws.xq + (size_t)t * H + (size_t)g * 8) = make_uint2(cw[0], cw[1]);
      const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
      for (int jj = 0; jj < k; ++jj)
        reinterpret_cast<uint4*>(ws.xh_perm + (size_t)pslot_s[tl][jj] * H)[g] = ov;
    }
    return;
  }
  const int sh = token_shift(fmaxf(am_s[tl][0], am_s[tl][1]));
  const float f = pow2f(-sh);
  if (q == 0) ws.xfac[t] = pow2f(sh);
  for (int g = q; g < H / 8; g += 64) {
    const uint4 u = reinterpret_cast<const uint4*>(x + (size_t)t * H)[g];
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 hh = __floats2half2_rn(__fmul_rn(bf16_lo(w4[i]), f), __fmul_rn(bf16_hi(w4[i]), f));
      o[i] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
    for (int jj = 0; jj < k; ++jj)
      reinterpret_cast<uint4*>(ws.xh_perm + (size_t)pslot_s[tl][jj] * H)[g] = ov;
  }
}

// h of every slot as the down operand by padded slot: f16(h * 2^-s), s from the slot's max |h|.
__global__ void __launch_bounds__(256) k_hprep16(WsView ws, int a8) {
  const int I = ws.I;
  const int j = blockIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  if (j >= (int)ws.ctl[kCtlTokenTiles]) return;
  const int slot0 = ws.tt_slot0[j], n = ws.tt_n[j];
  const int words = n * (I / 2);
  if (a8) {
    // W4A8: the E4M3 h codes' values (exact in f16); the scale is applied by the down GEMM
    for (int i = threadIdx.x; i < words; i += 256) {
      const int r = i / (I / 2), wd = i % (I / 2);
      const uint32_t two = *reinterpret_cast<const uint16_t*>(ws.hq + (size_t)(slot0 + r) * I +
                                                              2 * wd);
      reinterpret_cast<uint32_t*>(ws.hf_perm + ((size_t)j * 128 + r) * I)[wd] =
          e4m3x2_to_f16x2(two);
    }
    return;
  }
  for (int i = threadIdx.x; i < words; i += 256) {
    const int r = i / (I / 2), wd = i % (I / 2);
    const int sh = amax_shift(__uint_as_float(ws.slot_amax[slot0 + r]));
    const float f = pow2f(-sh);
    const uint32_t v = reinterpret_cast<const uint32_t*>(ws.h16 + (size_t)(slot0 + r) * I)[wd];
    const __half2 hh = __floats2half2_rn(__fmul_rn(__uint_as_float(v << 16), f),
                                         __fmul_rn(__uint_as_float(v & 0xFFFF0000u), f));
    reinterpret_cast<uint32_t*>(ws.hf_perm + ((size_t)j * 128 + r) * I)[wd] =
        *reinterpret_cast<const uint32_t*>(&hh);
  }
}

}  // namespace tc

// ------------------------------------------------------------------ host side
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D byte tensor [rows][row_bytes] with a box of box_bytes x box_rows (128-byte swizzle for
// 128-byte boxes, none for narrower ones).
bool make_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows,
              uint32_t box_rows, uint32_t box_bytes = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_bytes, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace

bool tc_supported() { return encode_fn() != nullptr; }

bool tile_path(int T, int H, int I, int mode) {
  if (T <= kNarrowT || !tc_supported()) return false;
  if (mode == 1) return H % 256 == 0 && I % 64 == 0;
  if (mode == 0 || mode == 2) return H % 128 == 0 && I % 128 == 0;   // kind::f16 (W4A16, W4A8)
  return false;
}

size_t tc_smem_bytes() { return (size_t)tc::kSmem; }

cudaError_t launch_tc_router(const LaunchCfg& lc, const uint16_t* x, const uint16_t* wr,
                             const WsView& ws) {
  CUtensorMap m_w, m_x;
  if (!make_map(&m_w, wr, (uint64_t)ws.H * 2, (uint64_t)ws.E, 128) ||
      !make_map(&m_x, x, (uint64_t)ws.H * 2, (uint64_t)ws.T, 128))
    return cudaErrorInvalidValue;
  const size_t smem = (size_t)tc::kRStages * 2 * tc::kTileBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(tc::k_tc_router, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int tiles = ((ws.E + 127) / 128) * ((ws.T + 127) / 128);
  const int grid = tiles < 2 * lc.num_sms ? tiles : 2 * lc.num_sms;
  return launch_kernel(lc, tc::k_tc_router, dim3(grid), dim3(tc::kRThreads), smem, m_w, m_x, ws);
}

cudaError_t launch_tc_experts(const LaunchCfg& lc, const PackView& pk, const WsView& ws,
                              const uint16_t* x, float xS, float x_inv6S) {
  const int H = pk.H, I = pk.I, E = pk.E;
  const uint64_t P = (uint64_t)ws.NT * 128;
  CUtensorMap m_gate, m_up, m_x, m_down, m_h;
  if (!make_map(&m_gate, pk.gate_codes, H / 2, (uint64_t)E * I, 16) ||
      !make_map(&m_up, pk.up_codes, H / 2, (uint64_t)E * I, 16) ||
      !make_map(&m_x, ws.xq_perm, H / 2, P, 128) ||
      !make_map(&m_down, pk.down_codes, I / 2, (uint64_t)E * H, 128) ||
      !make_map(&m_h, ws.hq_perm, I / 2, P, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_kernel(lc, tc::k_xquant_perm, dim3((ws.T + tc::kXqTok - 1) / tc::kXqTok),
                         dim3(64 * tc::kXqTok), 0, x, ws, xS, x_inv6S);
  if (e != cudaSuccess) return e;
  // one warp per (token tile, 16 atoms); the token-tile count is an upper bound read on the device
  const int xsf_warps = ws.NT * (H / 64 / 4);
  e = launch_kernel(lc, tc::k_xsf_atoms, dim3((xsf_warps + 7) / 8), dim3(256), 0, ws);
  if (e != cudaSuccess) return e;
  const size_t smem = tc_smem_bytes();
  e = cudaFuncSetAttribute(tc::k_tc_gemm<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc::k_tc_gemm<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  tc::TcParams pg;
  pg.sfa = pk.sfa_gu;
  pg.sfb = ws.xsf_atoms;
  pg.mult = pk.mult;
  pg.dscale = pk.down_in_scale;
  pg.dinv6 = pk.down_inv6S;
  pg.xS = xS;
  pg.H = H; pg.I = I; pg.E = E;
  pg.MT = I / 64;
  pg.nks = H / tc::kStageK;
  pg.last_k4 = 4;
  pg.a8 = 0;
  const int grid = tc::kCtasPerSm * lc.num_sms;   // persistent: two CTAs per SM
  e = launch_kernel(lc, tc::k_tc_gemm<false>, dim3(grid), dim3(tc::kThreads), smem, m_gate, m_up,
                    m_x, pg, ws);
  if (e != cudaSuccess) return e;
  tc::TcParams pd = pg;
  pd.sfa = pk.sfa_down;
  pd.sfb = ws.hsf_atoms;
  pd.MT = H / 128;
  pd.nks = (I + tc::kStageK - 1) / tc::kStageK;
  pd.last_k4 = ((I % tc::kStageK) ? (I % tc::kStageK) : tc::kStageK) / 64;
  // resident-h down GEMM when two h tiles, the Y staging and two weight tiles fit in shared memory
  pd.ustride = ((uint32_t)pd.nks * tc::kTileBytes + (uint32_t)(I / 64) * 512 + 1023u) & ~1023u;
  const int budget = 232448 - 2048 - tc::kRhStaging;
  const int nsw = (budget - 2 * (int)pd.ustride) / (int)pd.ustride;
  CUtensorMap m_y32, m_y16;
  if (I <= 1024 && nsw >= 2 &&
      make_map(&m_y32, ws.y, (uint64_t)H * 2, (uint64_t)ws.T * ws.k, 32) &&
      make_map(&m_y16, ws.y, (uint64_t)H * 2, (uint64_t)ws.T * ws.k, 16)) {
    pd.nsw = nsw < tc::kRhMaxStages ? nsw : tc::kRhMaxStages;
    const size_t smem_rd = (size_t)(2 + pd.nsw) * pd.ustride + tc::kRhStaging + 1024;
    e = cudaFuncSetAttribute(tc::k_tc_down, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_rd);
    if (e != cudaSuccess) return e;
    return launch_kernel(lc, tc::k_tc_down, dim3(lc.num_sms), dim3(tc::kThreads), smem_rd, m_down,
                         m_h, m_y32, m_y16, pd, ws);
  }
  return launch_kernel(lc, tc::k_tc_gemm<true>, dim3(grid), dim3(tc::kThreads), smem, m_down,
                       m_down, m_h, pd, ws);
}

}  // namespace moe

namespace moe {

cudaError_t launch_tc16_experts(const LaunchCfg& lc, const PackView& pk, const WsView& ws,
                                const uint16_t* x, int a8, float xS, float x_r8) {
  const int H = pk.H, I = pk.I, E = pk.E;
  const uint64_t P = (uint64_t)ws.NT * 128;
  CUtensorMap m_gate, m_up, m_x, m_down, m_h;
  if (!make_map(&m_gate, pk.gate_codes, H / 2, (uint64_t)E * I, 128, 32) ||
      !make_map(&m_up, pk.up_codes, H / 2, (uint64_t)E * I, 128, 32) ||
      !make_map(&m_x, ws.xh_perm, (uint64_t)H * 2, P, 128) ||
      !make_map(&m_down, pk.down_codes, I / 2, (uint64_t)E * H, 128, 32) ||
      !make_map(&m_h, ws.hf_perm, (uint64_t)I * 2, P, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_kernel(lc, tc::k_xprep16_perm, dim3((ws.T + tc::kXqTok - 1) / tc::kXqTok),
                         dim3(64 * tc::kXqTok), 0, x, ws, a8, xS, x_r8);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc::k_tc16<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           tc::T16<false>::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc::k_tc16<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           tc::T16<true>::kSmem);
  if (e != cudaSuccess) return e;
  tc::TcParams pg;
  pg.sfa = pk.sfa_gu;
  pg.sfb = nullptr;
  pg.mult = pk.mult;
  pg.dscale = pk.down_in_scale;
  pg.dinv6 = pk.down_inv6S;
  pg.xS = 1.0f;
  pg.H = H; pg.I = I; pg.E = E;
  pg.MT = I / 128;
  pg.nks = H / 64;
  pg.last_k4 = 0;
  pg.a8 = a8;
  const int grid = lc.num_sms;
  e = launch_kernel(lc, tc::k_tc16<false>, dim3(grid), dim3(tc::kT16Threads), tc::T16<false>::kSmem,
             m_gate, m_up, m_x, pg, ws);
  if (e != cudaSuccess) return e;
  e = launch_kernel(lc, tc::k_hprep16, dim3(ws.NT), dim3(256), 0, ws, a8);
  if (e != cudaSuccess) return e;
  tc::TcParams pd = pg;
  pd.sfa = pk.sfa_down;
  pd.MT = H / 128;
  pd.nks = I / 64;
  // the down GEMM with the h tile resident when it and two weight stages fit in shared memory
  const int abytes = (I / 64) * 16384;
  // Y through TMA boxes when their staging fits beside two load stages, else plain row stores
  const int room = 232448 - 2048 - abytes - tc::kDnConvBufs * tc::kDnConv;
  int ybox = (room - tc::kDnYStaging) / tc::kDnLStage >= 2 ? 1 : 0;
  int nst = (room - (ybox ? tc::kDnYStaging : 0)) / tc::kDnLStage;
  if (nst > tc::kDnMaxStages) nst = tc::kDnMaxStages;
  CUtensorMap m_y32, m_y16;
  if (ybox && !(make_map(&m_y32, ws.y, (uint64_t)H * 2, (uint64_t)ws.T * ws.k, 32) &&
                make_map(&m_y16, ws.y, (uint64_t)H * 2, (uint64_t)ws.T * ws.k, 16)))
    return cudaErrorInvalidValue;
  if (!ybox) m_y32 = m_y16 = m_down;   // not read
  if (H % tc::kDnN == 0 && nst >= 2) {
    const int smem = abytes + tc::kDnConvBufs * tc::kDnConv + nst * tc::kDnLStage +
                     (ybox ? tc::kDnYStaging : 0) + 1024;
    e = cudaFuncSetAttribute(tc::k_tc16_dn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(lc, tc::k_tc16_dn, dim3(grid), dim3(tc::kT16Threads), (size_t)smem, m_down, m_h,
                  m_y32, m_y16, pd, ws, nst, ybox);
  }
  return launch_kernel(lc, tc::k_tc16<true>, dim3(grid), dim3(tc::kT16Threads), tc::T16<true>::kSmem,
                m_down, m_down, m_h, pd, ws);
}

}  // namespace moe
