// moe_experts.cu — NVFP4 expert kernels of the routed-expert MoE step (sm_103a):
// gate/up with fused SiLU*up (and NVFP4 quantisation of h in W4A4), down, and the
// deterministic fixed-order combine.
//
// The expert matrices are NVFP4 (model card "Qwen3.8-Flash-Next NVIDIA NVFP4 for Infernix
// (bit-exact)", section "What is bit-exact and what is quantized": E2M1 codes, one E4M3 scale
// per 16 weights, FP32 multiplier and activation input scale per matrix). The release notes
// "Infernix windows-2026.10.11", section "Highlights", describe the sm_120a design these
// kernels replace: narrow calls of up to 8 columns on one-column kernels that convert FP4 to
// half2 in one instruction, and a down pass chained to gate/up with programmatic dependent
// launch. Here:
//   * One producer warp per CTA streams weight tiles HBM -> shared memory with TMA bulk copies
//     (cp.async.bulk) into a ring of stages guarded by mbarriers; consumer warps never issue
//     global loads for weights. Every wait is bounded.
//   * Consumers decode E2M1 -> f16x2 and E4M3 -> f16x2 with the hardware conversions
//     (code * scale is exact in f16) and multiply with m16n8k16 tensor-core MMAs, 8 tokens as N,
//     FP32 accumulation. Decode (<= 8 tokens) would otherwise be ALU-bound on CUDA cores.
//   * Tasks are (token group, row tile); groups hold <= 8 tokens of one expert, so the same
//     kernels serve decode (one group per expert) and the grouped prefill fallback.
#include "moe_internal.cuh"

#include <cuda_bf16.h>

namespace moe {
namespace {

constexpr int kGuConsumers = 8;
constexpr int kGuThreads = (kGuConsumers + 1) * 32;
constexpr int kDnConsumers = 4;
constexpr int kDnThreads = (kDnConsumers + 1) * 32;
constexpr int kMaxSmem = 232448;  // 227 KB opt-in per block

struct GuGeom {
  int KC;          // reduction columns per stage (== H when a whole task fits one stage)
  int nkc;         // stages per task (H / KC)
  int row_bytes;   // KC / 2: code bytes per row in a stage (rows packed, no padding)
  int stage_bytes; // 32 rows of codes + gate/up scales
  int stages;
  int x_stride;    // bytes per activation row in shared memory (2H + 64)
  int x_rows;      // T if resident else 8
  int tiles;       // I / 16
  int meta_cap;    // group records staged per CTA
};

struct DnGeom {
  int stage_bytes;  // 64 rows * I/2 codes + 4*I scales
  int stages;
  int h_stride;     // 2I + 16
  int h_rows;       // slots if resident else 8
  int tiles;        // H / 64
  int meta_cap;
  int raw_bytes;    // raw h staging area (resident h only)
};

constexpr int kMetaCap = 8;   // group records staged per CTA (a CTA's task range spans few groups)

GuGeom gu_geom(int H, int I, bool x_resident, int T) {
  GuGeom g;
  g.KC = H <= 4096 ? H : 4096;
  while (H % g.KC) g.KC -= 128;
  g.nkc = H / g.KC;
  g.row_bytes = g.KC / 2;
  g.stage_bytes = 32 * g.row_bytes + 2 * g.KC;
  g.x_stride = 2 * H + 64;
  g.x_rows = x_resident ? T : kGroup;
  g.tiles = I / 16;
  g.meta_cap = kMetaCap;
  const int fixed = g.x_rows * g.x_stride + kGuConsumers * 2 * 32 * 16 +
                    g.meta_cap * (int)sizeof(GroupMeta) + 1024;
  int st = (kMaxSmem - fixed) / g.stage_bytes;
  g.stages = st > 3 ? 3 : st;
  return g;
}

size_t gu_smem(const GuGeom& g) {
  return (size_t)g.stages * g.stage_bytes + (size_t)g.x_rows * g.x_stride +
         kGuConsumers * 2 * 32 * 16 + g.meta_cap * sizeof(GroupMeta) + 2 * 8 * g.stages + 64;
}

DnGeom dn_geom(int H, int I, bool h_resident, int slots, int mode) {
  DnGeom d;
  d.stage_bytes = 64 * (I / 2) + 4 * I;
  d.h_stride = 2 * I + 16;
  d.h_rows = h_resident ? slots : kGroup;
  d.tiles = H / 64;
  d.meta_cap = kMetaCap;
  const int raw = mode == 0 ? slots * I * 2 : slots * (I / 2) + ((slots * (I / 16) + 15) / 16) * 16;
  d.raw_bytes = h_resident ? raw : 0;
  const int fixed = d.h_rows * d.h_stride + d.raw_bytes + d.h_rows * 4 +
                    d.meta_cap * (int)sizeof(GroupMeta) + 1024;
  int st = (kMaxSmem - fixed) / d.stage_bytes;
  d.stages = st > 8 ? 8 : st;
  return d;
}

size_t dn_smem(const DnGeom& d) {
  return (size_t)d.stages * d.stage_bytes + (size_t)d.h_rows * d.h_stride + d.raw_bytes +
         d.h_rows * 4 + d.meta_cap * sizeof(GroupMeta) + 2 * 8 * d.stages + 64;
}

// Balanced contiguous task range of this CTA.
__device__ __forceinline__ void task_range(int ntasks, int& q0, int& q1) {
  q0 = (int)(((long long)ntasks * blockIdx.x) / gridDim.x);
  q1 = (int)(((long long)ntasks * (blockIdx.x + 1)) / gridDim.x);
}

// Stage the group records of groups [g0, g0 + n) into shared memory (n <= kMetaCap).
__device__ __forceinline__ void stage_meta(GroupMeta* dst, const GroupMeta* src, int g0, int n,
                                           int tid, int nthreads) {
  const int words = n * (int)(sizeof(GroupMeta) / 16);
  const uint4* s4 = reinterpret_cast<const uint4*>(src + g0);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (int i = tid; i < words; i += nthreads) d4[i] = s4[i];
}

// ------------------------------------------------------------------ gate/up
// grid: persistent, one CTA per SM; block: 8 consumer warps + 1 producer warp.
// A task is (token group gi, 16-row tile `it` of the intermediate dimension): gate and up rows
// it*16..+15 for the group's tokens over the full hidden dimension. The rows of a 16-row tile
// are contiguous in the pack, so a whole task is 4 TMA bulk copies (gate codes, up codes, gate
// scales, up scales) when it fits one stage.
__global__ void __launch_bounds__(kGuThreads, 1)
    k_gateup(PackView pk, WsView ws, GuGeom geo, int mode, int x_resident) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* stages = smem;
  unsigned char* xs = stages + (size_t)geo.stages * geo.stage_bytes;
  float* red = reinterpret_cast<float*>(xs + (size_t)geo.x_rows * geo.x_stride);
  GroupMeta* meta = reinterpret_cast<GroupMeta*>(red + kGuConsumers * 2 * 32 * 4);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + geo.meta_cap);
  uint64_t* empty = full + geo.stages;
  __shared__ volatile int abort_s;
  __shared__ int cur_group_s;
  __shared__ uint64_t xbar;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = pk.H, I = pk.I;
  if (tid == 0) {
    for (int s = 0; s < geo.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGuConsumers);
    }
    mbar_init(&xbar, 1);
    fence_mbar_init();
    abort_s = 0;
    cur_group_s = -1;
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();

  const int G = (int)ws.ctl[kCtlGroups];
  const int ntasks = G * geo.tiles;
  int q0, q1;
  task_range(ntasks, q0, q1);
  const int gfirst = q0 / geo.tiles;
  const int glast = q1 > q0 ? (q1 - 1) / geo.tiles : gfirst - 1;

  if (warp == kGuConsumers) {
    // ---------------- producer
    if (lane != 0) return;
    if (x_resident) {
      // the T activation rows (already in the permuted operand layout), one copy per row
      mbar_arrive_expect_tx(&xbar, (uint32_t)ws.T * H * 2);
      for (int t = 0; t < ws.T; ++t)
        bulk_g2s(xs + (size_t)t * geo.x_stride, ws.xh + (size_t)t * H, (uint32_t)H * 2, &xbar);
    }
    int chunk = 0;
    const uint32_t half = geo.row_bytes;
    for (int q = q0; q < q1 && !abort_s; ++q) {
      const int gi = q / geo.tiles, it = q % geo.tiles;
      const int e = __ldg(&ws.gmeta[gi].expert);
      const size_t row0 = (size_t)e * I + (size_t)it * 16;
      const uint8_t* gsrc = pk.gate_codes + row0 * (H / 2);
      const uint8_t* usrc = pk.up_codes + row0 * (H / 2);
      const uint8_t* gsc = pk.gu_scales + (((size_t)0 * pk.E + e) * geo.tiles + it) * (size_t)H;
      const uint8_t* usc = pk.gu_scales + (((size_t)1 * pk.E + e) * geo.tiles + it) * (size_t)H;
      for (int kc = 0; kc < geo.nkc; ++kc, ++chunk) {
        const int s = chunk % geo.stages, n = chunk / geo.stages;
        if (n > 0 && !mbar_wait(&empty[s], (n - 1) & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
          break;
        }
        unsigned char* st = stages + (size_t)s * geo.stage_bytes;
        mbar_arrive_expect_tx(&full[s], 32 * half + 2 * geo.KC);
        if (geo.nkc == 1) {
          bulk_g2s(st, gsrc, 16 * half, &full[s]);
          bulk_g2s(st + 16 * half, usrc, 16 * half, &full[s]);
        } else {
          for (int r = 0; r < 16; ++r) {
            bulk_g2s(st + r * half, gsrc + (size_t)r * (H / 2) + (size_t)kc * half, half, &full[s]);
            bulk_g2s(st + (16 + r) * half, usrc + (size_t)r * (H / 2) + (size_t)kc * half, half,
                     &full[s]);
          }
        }
        bulk_g2s(st + 32 * half, gsc + (size_t)kc * geo.KC, geo.KC, &full[s]);
        bulk_g2s(st + 32 * half + geo.KC, usc + (size_t)kc * geo.KC, geo.KC, &full[s]);
      }
    }
    // Do not leave while copies into this CTA's shared memory may still be in flight.
    const int used = chunk < geo.stages ? chunk : geo.stages;
    for (int i = 0; i < used; ++i) {
      const int c = chunk - 1 - i;
      (void)mbar_wait(&full[c % geo.stages], (c / geo.stages) & 1);
    }
    if (x_resident) (void)mbar_wait(&xbar, 0);
    return;
  }

  // ---------------- consumers
  const int g = lane >> 2, c = lane & 3;
  const int ncons = kGuConsumers * 32;
  const int nmeta = glast - gfirst + 1;
  if (nmeta > 0) stage_meta(meta, ws.gmeta, gfirst, nmeta < geo.meta_cap ? nmeta : geo.meta_cap,
                            tid, ncons);
  consumer_sync(ncons);
  if (x_resident && !mbar_wait(&xbar, 0)) {
    record_status(ws.ctl, kStTimeout);
    abort_s = 1;
  }
  int chunk = 0;
  const int jb_per_chunk = geo.KC / 128;
  for (int q = q0; q < q1; ++q) {
    const int gi = q / geo.tiles, it = q % geo.tiles;
    const int mi = gi - gfirst;
    const GroupMeta& gm = (mi < geo.meta_cap) ? meta[mi] : ws.gmeta[gi];
    const int slot0 = gm.slot0, n = gm.n;
    if (!x_resident && gi != cur_group_s) {
      consumer_sync(ncons);
      // the group's activation rows (already in the permuted operand layout), 4 loads in flight
      // per thread
      for (int i0 = tid; i0 < kGroup * (H / 8); i0 += 4 * ncons) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * ncons, r = i / (H / 8), w = i % (H / 8);
          v[u] = (i < kGroup * (H / 8) && r < n)
                     ? reinterpret_cast<const uint4*>(ws.xh + (size_t)ws.perm[slot0 + r] * H)[w]
                     : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * ncons, r = i / (H / 8), w = i % (H / 8);
          if (i < kGroup * (H / 8))
            *reinterpret_cast<uint4*>(xs + (size_t)r * geo.x_stride + w * 16) = v[u];
        }
      }
      consumer_sync(ncons);
      if (tid == 0) cur_group_s = gi;
    }
    const bool gvalid = g < n;
    const int xrow = x_resident ? (gvalid ? gm.tok[g] : 0) : g;
    const unsigned char* xr = xs + (size_t)xrow * geo.x_stride + c * 16;

    float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kc = 0; kc < geo.nkc; ++kc, ++chunk) {
      const int s = chunk % geo.stages, nn = chunk / geo.stages;
      if (!abort_s && !mbar_wait(&full[s], nn & 1)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
      }
      const unsigned char* st = stages + (size_t)s * geo.stage_bytes;
      const unsigned char* scb = st + 32 * geo.row_bytes + c * 32 + g * 4;
      for (int jb = warp; jb < jb_per_chunk; jb += kGuConsumers) {
        const int off = jb * 64 + c * 16;
        const uint4 gr = lds128(st + g * geo.row_bytes + off);
        const uint4 gr8 = lds128(st + (g + 8) * geo.row_bytes + off);
        const uint4 ur = lds128(st + (16 + g) * geo.row_bytes + off);
        const uint4 ur8 = lds128(st + (24 + g) * geo.row_bytes + off);
        const uint32_t scg = lds32(scb + jb * 128);
        const uint32_t scu = lds32(scb + geo.KC + jb * 128);
        uint4 xb[4];
        if (gvalid || !x_resident) {
          const unsigned char* xp = xr + (size_t)(kc * jb_per_chunk + jb) * 256;
#pragma unroll
          for (int p = 0; p < 4; ++p) xb[p] = lds128(xp + p * 64);
        } else {
#pragma unroll
          for (int p = 0; p < 4; ++p) xb[p] = make_uint4(0, 0, 0, 0);
        }
        kblock128_mma(accg, gr, gr8, scg, xb);
        kblock128_mma(accu, ur, ur8, scu, xb);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // fixed-order reduction over the consumer warps
    float* myred = red + (size_t)(warp * 2) * 32 * 4;
    *reinterpret_cast<float4*>(myred + lane * 4) = make_float4(accg[0], accg[1], accg[2], accg[3]);
    *reinterpret_cast<float4*>(myred + 128 + lane * 4) =
        make_float4(accu[0], accu[1], accu[2], accu[3]);
    consumer_sync(ncons);
    if (warp == 0) {
      float G4[4] = {0.f, 0.f, 0.f, 0.f}, U4[4] = {0.f, 0.f, 0.f, 0.f};
      for (int w = 0; w < kGuConsumers; ++w) {
        const float4 a = *reinterpret_cast<const float4*>(red + (size_t)(w * 2) * 128 + lane * 4);
        const float4 b =
            *reinterpret_cast<const float4*>(red + (size_t)(w * 2) * 128 + 128 + lane * 4);
        G4[0] += a.x; G4[1] += a.y; G4[2] += a.z; G4[3] += a.w;
        U4[0] += b.x; U4[1] += b.y; U4[2] += b.z; U4[3] += b.w;
      }
      float hv[4];  // (row g, col 2c), (row g, col 2c+1), (row g+8, col 2c), (row g+8, col 2c+1)
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        const int col = 2 * c + (q2 & 1);
        const int tok = col < n ? (x_resident ? gm.tok[col] : ws.perm[slot0 + col]) : 0;
        const float xf = col < n ? ws.xfac[tok] : 0.0f;
        const float gv = G4[q2] * gm.mg * xf;
        const float uv = U4[q2] * gm.mu * xf;
        hv[q2] = col < n ? silu_mul(gv, uv) : 0.0f;
      }
      const int i0 = it * 16 + g;
      if (mode == 0) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int col = 2 * c + cc;
          const uint16_t b0 = f32_to_bf16_rn(hv[cc]), b1 = f32_to_bf16_rn(hv[2 + cc]);
          // |h| of the BF16 values, for the down stage's per-slot f16 scaling
          float a = fmaxf(fabsf(__uint_as_float((uint32_t)b0 << 16)),
                          fabsf(__uint_as_float((uint32_t)b1 << 16)));
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
          if (col < n) {
            const size_t slot = (size_t)(slot0 + col);
            ws.h16[slot * I + i0] = b0;
            ws.h16[slot * I + i0 + 8] = b1;
            if (g == 0) atomicMax(&ws.slot_amax[slot], __float_as_uint(a));
          }
        }
      } else {
        const float Sd = gm.sd, i6 = gm.i6d;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {  // token column 2c + cc
          const float v_lo = hv[cc], v_hi = hv[2 + cc];  // elements g and g+8 of the block
          float a = fmaxf(fabsf(v_lo), fabsf(v_hi));
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
          const uint32_t sf = e4m3_encode_rn(__fmul_rn(a, i6));
          uint32_t lo = 0, hi = 0;
          if (sf != 0u) {
            const float r = __frcp_rn(__fmul_rn(e4m3_value_nonneg(sf), Sd));
            lo = e2m1_encode_rn(__fmul_rn(v_lo, r)) << (4 * g);  // elements 0..7 -> word 0
            hi = e2m1_encode_rn(__fmul_rn(v_hi, r)) << (4 * g);  // elements 8..15 -> word 1
          }
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            lo |= __shfl_xor_sync(0xFFFFFFFFu, lo, off);
            hi |= __shfl_xor_sync(0xFFFFFFFFu, hi, off);
          }
          const int col = 2 * c + cc;
          if (g == 0 && col < n) {
            const size_t slot = (size_t)(slot0 + col);
            *reinterpret_cast<uint2*>(ws.hq + slot * (I / 2) + it * 8) = make_uint2(lo, hi);
            ws.hsf[slot * (I / 16) + it] = static_cast<uint8_t>(sf);
          }
        }
      }
    }
    consumer_sync(ncons);
  }
}

// ------------------------------------------------------------------ down
// A task is (token group gi, 64-row tile ht of the hidden dimension); consumer warp w owns
// rows ht*64 + 16w .. +15. Y (BF16) goes to the slot-major buffer for the combine.
__global__ void __launch_bounds__(kDnThreads, 1)
    k_down(PackView pk, WsView ws, DnGeom geo, int mode, int h_resident) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* stages = smem;
  unsigned char* hs = stages + (size_t)geo.stages * geo.stage_bytes;
  unsigned char* raw = hs + (size_t)geo.h_rows * geo.h_stride;
  float* hfac = reinterpret_cast<float*>(raw + geo.raw_bytes);
  GroupMeta* meta = reinterpret_cast<GroupMeta*>(hfac + geo.h_rows + ((4 - (geo.h_rows & 3)) & 3));
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + geo.meta_cap);
  uint64_t* empty = full + geo.stages;
  __shared__ volatile int abort_s;
  __shared__ int cur_group_s;
  __shared__ uint64_t hbar;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = pk.H, I = pk.I;
  if (tid == 0) {
    for (int s = 0; s < geo.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDnConsumers);
    }
    mbar_init(&hbar, 1);
    fence_mbar_init();
    abort_s = 0;
    cur_group_s = -1;
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();

  const int G = (int)ws.ctl[kCtlGroups];
  const int ntasks = G * geo.tiles;
  int q0, q1;
  task_range(ntasks, q0, q1);
  const uint32_t code_bytes = 64u * (I / 2);
  const int gfirst = q0 / geo.tiles;
  const int glast = q1 > q0 ? (q1 - 1) / geo.tiles : gfirst - 1;

  const int S = ws.T * ws.k;
  if (warp == kDnConsumers) {
    if (lane != 0) return;
    if (h_resident) {
      // every slot's raw h in one or two copies (W4A16: BF16 rows; W4A4: codes, then scales)
      if (mode == 0) {
        mbar_arrive_expect_tx(&hbar, (uint32_t)S * I * 2);
        bulk_g2s(raw, ws.h16, (uint32_t)S * I * 2, &hbar);
      } else {
        const uint32_t cb = (uint32_t)S * (I / 2);
        const uint32_t sb = (uint32_t)((S * (I / 16) + 15) / 16) * 16;
        mbar_arrive_expect_tx(&hbar, cb + sb);
        bulk_g2s(raw, ws.hq, cb, &hbar);
        bulk_g2s(raw + cb, ws.hsf, sb, &hbar);
      }
    }
    int chunk = 0;
    for (int q = q0; q < q1 && !abort_s; ++q, ++chunk) {
      const int gi = q / geo.tiles, ht = q % geo.tiles;
      const int e = __ldg(&ws.gmeta[gi].expert);
      const int s = chunk % geo.stages, n = chunk / geo.stages;
      if (n > 0 && !mbar_wait(&empty[s], (n - 1) & 1)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
        break;
      }
      unsigned char* st = stages + (size_t)s * geo.stage_bytes;
      mbar_arrive_expect_tx(&full[s], code_bytes + 4u * I);
      bulk_g2s(st, pk.down_codes + ((size_t)e * H + (size_t)ht * 64) * (I / 2), code_bytes,
               &full[s]);
      bulk_g2s(st + code_bytes, pk.down_scales + ((size_t)e * geo.tiles + ht) * (4 * (size_t)I),
               4u * I, &full[s]);
    }
    const int used = chunk < geo.stages ? chunk : geo.stages;
    for (int i = 0; i < used; ++i) {
      const int c2 = chunk - 1 - i;
      (void)mbar_wait(&full[c2 % geo.stages], (c2 / geo.stages) & 1);
    }
    if (h_resident) (void)mbar_wait(&hbar, 0);
    return;
  }

  const int g = lane >> 2, c = lane & 3;
  const int ncons = kDnConsumers * 32;
  const int nmeta = glast - gfirst + 1;
  if (nmeta > 0) stage_meta(meta, ws.gmeta, gfirst, nmeta < geo.meta_cap ? nmeta : geo.meta_cap,
                            tid, ncons);
  // Stage h as the f16 operand: per-row factors first, then every (row, word) in one sweep so
  // that all loads are in flight together.
  auto row_factor = [&](int row, int slot, float sd) {
    if (mode == 0) {
      // BF16 h scaled by 2^-s puts the slot's amax in [2^14, 2^15): exact in f16
      hfac[row] = __int_as_float((127 + amax_shift(__uint_as_float(ws.slot_amax[slot]))) << 23);
    } else {
      hfac[row] = sd;
    }
  };
  auto stage_word = [&](int row, int slot, int i) {
    unsigned char* dst = hs + (size_t)row * geo.h_stride + i * 4;
    if (mode == 0) {
      const float f = 1.0f / hfac[row];  // exact: a power of two
      const uint32_t v = reinterpret_cast<const uint32_t*>(ws.h16 + (size_t)slot * I)[i];
      *reinterpret_cast<__half2*>(dst) =
          __floats2half2_rn(__fmul_rn(__uint_as_float(v << 16), f),
                            __fmul_rn(__uint_as_float(v & 0xFFFF0000u), f));
    } else {
      const uint32_t byte = ws.hq[(size_t)slot * (I / 2) + i];
      const float sv = e4m3_value_nonneg(ws.hsf[(size_t)slot * (I / 16) + i / 8]);
      *reinterpret_cast<__half2*>(dst) =
          __floats2half2_rn(e2m1_value(byte & 0xF) * sv, e2m1_value(byte >> 4) * sv);
    }
  };
  if (h_resident) {
    for (int gi = tid; gi < G; gi += ncons) {
      const GroupMeta& gm = ws.gmeta[gi];
      const int s0 = gm.slot0, nn = gm.n;
      const float sd = gm.sd;
      for (int r = 0; r < nn; ++r) row_factor(s0 + r, s0 + r, sd);
    }
    if (!mbar_wait(&hbar, 0)) {
      record_status(ws.ctl, kStTimeout);
      abort_s = 1;
    }
    consumer_sync(ncons);
    // convert the raw copy to the f16 operand rows, shared memory to shared memory
    for (int i = tid; i < S * (I / 2); i += ncons) {
      const int row = i / (I / 2), w = i % (I / 2);
      unsigned char* dst = hs + (size_t)row * geo.h_stride + w * 4;
      if (mode == 0) {
        const float f = 1.0f / hfac[row];  // exact: a power of two
        const uint32_t v = reinterpret_cast<const uint32_t*>(raw)[i];
        *reinterpret_cast<__half2*>(dst) =
            __floats2half2_rn(__fmul_rn(__uint_as_float(v << 16), f),
                              __fmul_rn(__uint_as_float(v & 0xFFFF0000u), f));
      } else {
        const uint32_t byte = raw[i];
        const float sv = e4m3_value_nonneg(raw[(size_t)S * (I / 2) + (size_t)row * (I / 16) + w / 8]);
        *reinterpret_cast<__half2*>(dst) =
            __floats2half2_rn(e2m1_value(byte & 0xF) * sv, e2m1_value(byte >> 4) * sv);
      }
    }
  }
  consumer_sync(ncons);
  int chunk = 0;
  for (int q = q0; q < q1; ++q, ++chunk) {
    const int gi = q / geo.tiles, ht = q % geo.tiles;
    const int mi = gi - gfirst;
    const GroupMeta& gm = (mi < geo.meta_cap) ? meta[mi] : ws.gmeta[gi];
    const int slot0 = gm.slot0, n = gm.n;
    if (!h_resident && gi != cur_group_s) {
      consumer_sync(ncons);
      if (tid < n) row_factor(tid, slot0 + tid, gm.sd);
      consumer_sync(ncons);
      for (int i = tid; i < n * (I / 2); i += ncons)
        stage_word(i / (I / 2), slot0 + i / (I / 2), i % (I / 2));
      consumer_sync(ncons);
      if (tid == 0) cur_group_s = gi;
    }
    const int s = chunk % geo.stages, nn = chunk / geo.stages;
    if (!abort_s && !mbar_wait(&full[s], nn & 1)) {
      record_status(ws.ctl, kStTimeout);
      abort_s = 1;
    }
    const unsigned char* st = stages + (size_t)s * geo.stage_bytes;
    const bool gvalid = g < n;
    const int hrow = h_resident ? slot0 + (gvalid ? g : 0) : g;
    const unsigned char* hr = hs + (size_t)hrow * geo.h_stride + c * 32;
    const int nkb = I / 64;
    const unsigned char* rg = st + (size_t)(warp * 16 + g) * (I / 2) + c * 8;
    const unsigned char* rg8 = rg + 8 * (I / 2);
    const unsigned char* scb = st + code_bytes + (size_t)warp * nkb * 64 + c * 16 + g * 2;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < nkb; ++j) {
      const uint2 a0 = lds64(rg + j * 32);
      const uint2 a1 = lds64(rg8 + j * 32);
      const uint32_t sc = lds16(scb + j * 64);
      uint4 xb0 = make_uint4(0, 0, 0, 0), xb1 = xb0;
      if (gvalid) {
        xb0 = lds128(hr + j * 128);
        xb1 = lds128(hr + j * 128 + 16);
      }
      kblock_mma(acc, a0, a1, sc, xb0, xb1);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    const float md = gm.md;
#pragma unroll
    for (int q2 = 0; q2 < 4; ++q2) {
      const int col = 2 * c + (q2 & 1);
      if (col < n) {
        const int hsrow = h_resident ? slot0 + col : col;
        const float y = acc[q2] * md * hfac[hsrow];
        const int row = ht * 64 + warp * 16 + g + ((q2 >> 1) << 3);
        ws.y[(size_t)(slot0 + col) * H + row] = f32_to_bf16_rn(y);
      }
    }
  }
}

// ------------------------------------------------------------------ combine
// out[t][r] = BF16( sum_{j=0..k-1} w[t][j] * Y[slot_of[t][j]][r] ), FP32, j in rank order.
// All k weight/slot loads are issued before the Y loads (no dependent load chain per j).

__global__ void __launch_bounds__(256) k_combine(WsView ws, uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const int H = ws.H, k = ws.k;
  const long long n8 = (long long)ws.T * (H / 8);
  for (long long it = (long long)blockIdx.x * 256 + threadIdx.x; it < n8;
       it += (long long)gridDim.x * 256) {
    const int t = (int)(it / (H / 8)), r8 = (int)(it % (H / 8));
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < k; j0 += 8) {
      // the weights and slots of 8 ranks, then their 8 Y loads, all issued before use
      float wj[8];
      int sj[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const bool ok = j0 + q < k;
        wj[q] = ok ? ws.w[(size_t)t * k + j0 + q] : 0.0f;
        sj[q] = ok ? ws.slot_of[(size_t)t * k + j0 + q] : -1;
      }
      uint4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        v[q] = sj[q] >= 0 ? reinterpret_cast<const uint4*>(ws.y + (size_t)sj[q] * H)[r8]
                          : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (sj[q] < 0) break;   // ranks in order: stop at the first past k
        const uint32_t wd[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          acc[2 * u] += wj[q] * __uint_as_float(wd[u] << 16);
          acc[2 * u + 1] += wj[q] * __uint_as_float(wd[u] & 0xFFFF0000u);
        }
      }
    }
    if (ws.sh_y) {
      // the shared expert's term, after the routed ones: sigma_t * BF16(Ys) (Ys is an expert
      // output, rounded to BF16 like the routed Y)
      const float sg = __ldcg(ws.sh_sigma + t);
      const float4* ys = reinterpret_cast<const float4*>(ws.sh_y + (size_t)t * H) + 2 * r8;
      const float4 a = __ldcg(ys), b = __ldcg(ys + 1);
      const float yv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += sg * bf16_round(yv[q]);
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = (uint32_t)f32_to_bf16_rn(acc[2 * q]) | ((uint32_t)f32_to_bf16_rn(acc[2 * q + 1]) << 16);
    reinterpret_cast<uint4*>(out + (size_t)t * H)[r8] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ------------------------------------------------------------------ residual sum
// out[i] = BF16(a[i] + b[i]): the next input of a chained layer (its input plus its output).
__global__ void __launch_bounds__(256) k_residual_add(const uint16_t* __restrict__ a,
                                                     const uint16_t* __restrict__ b,
                                                     uint16_t* __restrict__ out, size_t n8) {
  pdl_wait();
  pdl_launch_dependents();
  for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < n8; i += (size_t)gridDim.x * 256) {
    const uint4 va = __ldcg(reinterpret_cast<const uint4*>(a) + i);
    const uint4 vb = __ldcg(reinterpret_cast<const uint4*>(b) + i);
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = (uint32_t)f32_to_bf16_rn(bf16_lo(wa[q]) + bf16_lo(wb[q])) |
             ((uint32_t)f32_to_bf16_rn(bf16_hi(wa[q]) + bf16_hi(wb[q])) << 16);
    reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ------------------------------------------------------------------ scale re-layout
// checkpoint [E][rows][cols/16] -> fragment order (see PackView).
__global__ void k_pack_scales(const uint8_t* __restrict__ rg, const uint8_t* __restrict__ ru,
                              const uint8_t* __restrict__ rd, int E, int H, int I,
                              uint8_t* __restrict__ gu, uint8_t* __restrict__ dn, int inverse,
                              int only_expert, int only_which, uint8_t* __restrict__ raw_out) {
  // gate/up part: index over [mat][E][I/16][H/64][4][8][2]
  const long long n_gu = 2ll * E * I * (H / 16);
  const long long n_dn = (long long)E * H * (I / 16);
  for (long long o = (long long)blockIdx.x * blockDim.x + threadIdx.x; o < n_gu + n_dn;
       o += (long long)gridDim.x * blockDim.x) {
    if (o < n_gu) {
      // [mat][E][I/16][H/128][c 4][g 8][4]: byte 2h + b = row 16*tile + g + 8h, block 8J+2c+b
      long long r = o;
      const int b = (int)(r & 1); r >>= 1;
      const int h = (int)(r & 1); r >>= 1;
      const int g = (int)(r & 7); r >>= 3;
      const int c = (int)(r & 3); r >>= 2;
      const int J = (int)(r % (H / 128)); r /= (H / 128);
      const int tile = (int)(r % (I / 16)); r /= (I / 16);
      const int e = (int)(r % E); r /= E;
      const int mat = (int)r;
      const int row = tile * 16 + g + 8 * h;
      const int blk = 8 * J + 2 * c + b;
      const size_t src = ((size_t)e * I + row) * (H / 16) + blk;
      if (!inverse) {
        gu[o] = (mat == 0 ? rg : ru)[src];
      } else if (e == only_expert && mat == only_which) {
        raw_out[(size_t)row * (H / 16) + blk] = gu[o];
      }
    } else {
      long long r = o - n_gu;
      const int h = (int)(r & 1); r >>= 1;
      const int g = (int)(r & 7); r >>= 3;
      const int c = (int)(r & 3); r >>= 2;
      const int j = (int)(r % (I / 64)); r /= (I / 64);
      const int mt = (int)(r & 3); r >>= 2;
      const int ht = (int)(r % (H / 64)); r /= (H / 64);
      const int e = (int)r;
      const int row = ht * 64 + mt * 16 + g + 8 * h;
      const int blk = 4 * j + c;
      const size_t src = ((size_t)e * H + row) * (I / 16) + blk;
      if (!inverse) {
        dn[o - n_gu] = rd[src];
      } else if (e == only_expert && only_which == 2) {
        raw_out[(size_t)row * (I / 16) + blk] = dn[o - n_gu];
      }
    }
  }
}

// checkpoint scales -> tensor-core scale-factor atoms (see PackView).
__global__ void k_pack_sf_atoms(const uint8_t* __restrict__ rg, const uint8_t* __restrict__ ru,
                                const uint8_t* __restrict__ rd, int E, int H, int I,
                                uint8_t* __restrict__ at_gu, uint8_t* __restrict__ at_dn) {
  const long long n_gu = (long long)E * (I / 64) * (H / 64) * 512;
  const long long n_dn = (long long)E * (H / 128) * (I / 64) * 512;
  for (long long o = (long long)blockIdx.x * blockDim.x + threadIdx.x; o < n_gu + n_dn;
       o += (long long)gridDim.x * blockDim.x) {
    const bool gu = o < n_gu;
    long long q = gu ? o : o - n_gu;
    const int byte = (int)(q & 511); q >>= 9;
    const int r = (byte >> 4) + 32 * ((byte & 15) >> 2);   // row inside the 128-row tile
    const int b = byte & 3;                                // block inside the K step
    if (gu) {
      const int ks = (int)(q % (H / 64)); q /= (H / 64);
      const int mt = (int)(q % (I / 64)); q /= (I / 64);
      const int e = (int)q;
      // rows of the atom: the 64 gate and 64 up rows of intermediate tile mt interleaved by 16
      // (atom rows 32q .. 32q+15: gate rows mt*64 + 16q .., 32q+16 .. 32q+31: the up rows)
      const int row = mt * 64 + (r >> 5) * 16 + (r & 15);
      const uint8_t* src = (r & 16) ? ru : rg;
      at_gu[o] = src[((size_t)e * I + row) * (H / 16) + ks * 4 + b];
    } else {
      const int ks = (int)(q % (I / 64)); q /= (I / 64);
      const int mt = (int)(q % (H / 128)); q /= (H / 128);
      const int e = (int)q;
      const int row = mt * 128 + r;
      at_dn[o - n_gu] = rd[((size_t)e * H + row) * (I / 16) + ks * 4 + b];
    }
  }
}


}  // namespace

size_t gateup_smem_bytes(int H, bool x_resident, int T) {
  return gu_smem(gu_geom(H, 64, x_resident, T));
}

size_t down_smem_bytes(int I, bool h_resident, int slots) {
  return dn_smem(dn_geom(64, I, h_resident, slots, 0));
}

cudaError_t launch_gateup(const LaunchCfg& lc, const PackView& pk, const WsView& ws, int mode,
                          bool x_resident) {
  const GuGeom geo = gu_geom(pk.H, pk.I, x_resident, ws.T);
  if (geo.stages < 1) return cudaErrorInvalidConfiguration;
  const size_t smem = gu_smem(geo);
  cudaError_t e =
      cudaFuncSetAttribute(k_gateup, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int max_tasks = ws.G * geo.tiles;
  int grid = lc.num_sms < max_tasks ? lc.num_sms : max_tasks;
  if (grid < 1) grid = 1;
  return launch_kernel(lc, k_gateup, dim3(grid), dim3(kGuThreads), smem, pk, ws, geo, mode,
                x_resident ? 1 : 0);
}

cudaError_t launch_down(const LaunchCfg& lc, const PackView& pk, const WsView& ws, int mode,
                        bool h_resident) {
  DnGeom geo = dn_geom(pk.H, pk.I, h_resident, ws.T * ws.k, mode);
  if (h_resident && geo.stages < 2) {  // not enough room to keep every slot's h: stage per group
    h_resident = false;
    geo = dn_geom(pk.H, pk.I, false, ws.T * ws.k, mode);
  }
  if (geo.stages < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = dn_smem(geo);
  cudaError_t e =
      cudaFuncSetAttribute(k_down, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int max_tasks = ws.G * geo.tiles;
  int grid = lc.num_sms < max_tasks ? lc.num_sms : max_tasks;
  if (grid < 1) grid = 1;
  return launch_kernel(lc, k_down, dim3(grid), dim3(kDnThreads), smem, pk, ws, geo, mode,
                h_resident ? 1 : 0);
}

cudaError_t launch_combine(const LaunchCfg& lc, const WsView& ws, uint16_t* out) {
  const long long n8 = (long long)ws.T * (ws.H / 8);
  long long grid = (n8 + 255) / 256;
  const long long cap = (long long)lc.num_sms * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  return launch_kernel(lc, k_combine, dim3((unsigned)grid), dim3(256), 0, ws, out);
}

cudaError_t launch_residual_add(const LaunchCfg& lc, const uint16_t* a, const uint16_t* b,
                                uint16_t* out, size_t n) {
  const size_t n8 = n / 8;
  const unsigned grid = (unsigned)((n8 + 255) / 256 < (size_t)4 * lc.num_sms
                                       ? (n8 + 255) / 256 : (size_t)4 * lc.num_sms);
  return launch_kernel(lc, k_residual_add, dim3(grid > 0 ? grid : 1), dim3(256), 0, a, b, out, n8);
}

cudaError_t launch_pack_scales(cudaStream_t s, const uint8_t* raw_gate, const uint8_t* raw_up,
                               const uint8_t* raw_down, int E, int H, int I, uint8_t* gu_scales,
                               uint8_t* down_scales, uint8_t* sfa_gu, uint8_t* sfa_down) {
  k_pack_scales<<<1024, 256, 0, s>>>(raw_gate, raw_up, raw_down, E, H, I, gu_scales, down_scales,
                                     0, -1, -1, nullptr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || H % 128) return e;
  k_pack_sf_atoms<<<1024, 256, 0, s>>>(raw_gate, raw_up, raw_down, E, H, I, sfa_gu, sfa_down);
  return cudaGetLastError();
}

cudaError_t launch_unpack_scales(cudaStream_t s, const uint8_t* gu_scales,
                                 const uint8_t* down_scales, int E, int H, int I, int expert,
                                 int which, uint8_t* raw_out) {
  k_pack_scales<<<1024, 256, 0, s>>>(nullptr, nullptr, nullptr, E, H, I,
                                     const_cast<uint8_t*>(gu_scales),
                                     const_cast<uint8_t*>(down_scales), 1, expert, which, raw_out);
  return cudaGetLastError();
}

}  // namespace moe
