// moe_decode.cu — the whole routed-expert MoE step of a narrow call (T <= 8 tokens: decode and
// speculative verification) in ONE persistent kernel on sm_103a.
//
// The pages' engine runs this step as a chain of small kernels joined by programmatic dependent
// launch (release notes "Infernix windows-2026.10.11", section "Highlights"). At one token the
// step moves ~26 MB, about 4 us of HBM time, while every kernel boundary costs a few
// microseconds of drain, launch and first-copy latency. Here one CTA per SM runs every phase,
// and CTAs meet only at two grid-wide barriers (bounded spins on counters in the workspace):
//
//   1. router: each CTA copies its 3-4 router rows (TMA bulk copy, issued before waiting for
//      the preceding kernel: the router does not depend on it) and the T activation rows, and
//      writes its logits.                                                    -> barrier 1
//      While waiting, each CTA converts the activations into the f16 (W4A16) or NVFP4-decoded
//      (W4A4) MMA operand in its own shared memory, and writes its share of the W4A4 codes.
//   2. routing: every CTA selects the top-k of every token itself (one warp per token) and
//      builds the expert groups in shared memory; no second barrier is needed. CTA 0 publishes
//      idx / w / counts / offsets / perm / slot_of.
//   3. gate/up + SiLU*up: tasks (group, 16-row tile of I), as in the multi-kernel path.
//      As soon as its last gate/up stage is free, the producer warp streams this CTA's down
//      weights into the same shared memory, so they load while h is finished elsewhere.
//                                                                            -> barrier 2
//   4. down: tasks (group, 128-row tile of H); each task writes Y (BF16). The CTA that finishes
//      the last task of a 128-row tile (a ticket per tile) forms out for those rows: the
//      fixed-order weighted sum over each token's k experts (rank order, FP32, then BF16).
//
// Every product, rounding and summation order is the one of the multi-kernel path.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kDcWarps = 8;                       // consumer warps
constexpr int kDcThreads = (kDcWarps + 1) * 32;   // + one producer warp
constexpr int kDcCons = kDcWarps * 32;
constexpr int kDnRows = 128;                      // rows of H per down task (16 per warp)
constexpr int kDcSmemMax = 232448;                // 227 KB opt-in per block
constexpr int kDcStatic = 512;                    // static shared memory allowance

// One expert's token group (<= 8 tokens) of the current call.
struct DcGroup {
  int expert, slot0, n;
  uint32_t toks;          // token of column c in bits 4c .. 4c+3
  float mg, mu, md, sd;   // gate/up/down multipliers, down input scale
  float i6d;              // fl32(1 / fl32(6 * sd))
  int pad[3];
};
static_assert(sizeof(DcGroup) == 48, "DcGroup layout");

struct DcGeom {
  int rows_max;                 // router rows of one CTA, at most
  int wpr;                      // warps per router row (2: each warp half a row)
  int KC, nkc, row_bytes;       // gate/up stage: KC reduction columns, nkc stages per task
  int gu_stage, gu_stages;
  int dn_stage, dn_stages;
  int arena;                    // router rows + raw x | routing scratch | gate/up ring | down ring
  int x_stride;                 // 2H + 64: one x operand row
  int h_stride;                 // 2I + 16: one h operand row
  int xop;                      // x operand rows, later the h operand rows of one group
  int smax, gmax;               // slots T*k, groups min(T*k, E)
  int smem;
};

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier halves (thread 0 of the CTA; the callers synchronise the CTA around them).
__device__ __forceinline__ void grid_arrive(uint32_t* ctr) {
  __threadfence();
  atomicAdd(ctr, 1u);
}
__device__ __forceinline__ bool grid_wait(const uint32_t* ctr, uint32_t target) {
  if (ld_acquire(ctr) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 16; ++i)
      if (ld_acquire(ctr) >= target) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ int group_tok(uint32_t toks, int c) { return (toks >> (4 * c)) & 0xF; }

// Exclusive scan of a[0..n) in place by one warp; returns the total.
__device__ __forceinline__ int warp_exclusive_scan(int32_t* a, int n, int lane) {
  const int per = (n + 31) / 32;
  const int b0 = lane * per, b1 = min(n, b0 + per);
  int s = 0;
  for (int i = b0; i < b1; ++i) s += a[i];
  int incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  int run = incl - s;
  for (int i = b0; i < b1; ++i) {
    const int v = a[i];
    a[i] = run;
    run += v;
  }
  return __shfl_sync(0xFFFFFFFFu, incl, 31);
}

__device__ __forceinline__ void balanced_range(int ntasks, int& q0, int& q1) {
  q0 = (int)(((long long)ntasks * blockIdx.x) / gridDim.x);
  q1 = (int)(((long long)ntasks * (blockIdx.x + 1)) / gridDim.x);
}

__global__ void __launch_bounds__(kDcThreads, 1)
    k_decode(PackView pk, WsView ws, DcGeom geo, const uint16_t* __restrict__ x,
             const uint16_t* __restrict__ wr, int mode, float xS, float x_inv6S,
             uint16_t* __restrict__ out) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* arena = smem;
  unsigned char* xop = arena + geo.arena;
  float* red = reinterpret_cast<float*>(xop + geo.xop);                 // [8 warps][2][128]
  DcGroup* grp = reinterpret_cast<DcGroup*>(red + kDcWarps * 2 * 128);
  int32_t* sel_idx = reinterpret_cast<int32_t*>(grp + geo.gmax);        // [S]
  float* sel_w = reinterpret_cast<float*>(sel_idx + geo.smax);          // [S]
  int32_t* sel_slot = reinterpret_cast<int32_t*>(sel_w + geo.smax);     // [S]
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(sel_slot + geo.smax) + 7) & ~uintptr_t(7));
  uint64_t* gfull = bars;
  uint64_t* gempty = gfull + geo.gu_stages;
  uint64_t* dfull = gempty + geo.gu_stages;
  uint64_t* dempty = dfull + geo.dn_stages;
  uint64_t* rbar = dempty + geo.dn_stages;
  uint64_t* xbar = rbar + 1;
  __shared__ float xfac_s[kNarrowT];
  __shared__ int shift_s[kNarrowT];
  __shared__ float hfac_s[kGroup], hinv_s[kGroup];
  __shared__ int U_s, last_s;
  __shared__ volatile int abort_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = ws.T, H = ws.H, E = ws.E, k = ws.k, I = ws.I, S = T * k;
  const int G = gridDim.x, b = blockIdx.x;
  const int row0 = (int)(((long long)E * b) / G);
  const int nrows = (int)(((long long)E * (b + 1)) / G) - row0;
  uint16_t* wrs = reinterpret_cast<uint16_t*>(arena);                            // [rows][H]
  uint16_t* xraw = reinterpret_cast<uint16_t*>(arena + (size_t)geo.rows_max * H * 2);  // [T][H]

  if (tid == 0) {
    for (int s = 0; s < geo.gu_stages; ++s) {
      mbar_init(&gfull[s], 1);
      mbar_init(&gempty[s], kDcWarps);
    }
    for (int s = 0; s < geo.dn_stages; ++s) {
      mbar_init(&dfull[s], 1);
      mbar_init(&dempty[s], kDcWarps);
    }
    mbar_init(rbar, 1);
    mbar_init(xbar, 1);
    fence_mbar_init();
    abort_s = 0;
    // the router rows are weights: copy them before waiting for the preceding kernel
    if (nrows > 0) {
      mbar_arrive_expect_tx(rbar, (uint32_t)nrows * H * 2);
      bulk_g2s(wrs, wr + (size_t)row0 * H, (uint32_t)nrows * H * 2, rbar);
    }
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (tid == 0) {
    mbar_arrive_expect_tx(xbar, (uint32_t)T * H * 2);
    bulk_g2s(xraw, x, (uint32_t)T * H * 2, xbar);
  }
  if (b == 0 && mode == 0)
    for (int i = tid; i < S; i += kDcThreads) ws.slot_amax[i] = 0u;
  if ((nrows > 0 && !mbar_wait(rbar, 0)) || !mbar_wait(xbar, 0)) {
    record_status(ws.ctl, kStTimeout);
    abort_s = 1;
  }

  // ---------------- 1. router rows (warps 0..7; warp w: row w / wpr, part w % wpr of H)
  if (warp < kDcWarps) {
    const int r = warp / geo.wpr, part = warp % geo.wpr;
    float acc[kNarrowT];
#pragma unroll
    for (int t = 0; t < kNarrowT; ++t) acc[t] = 0.0f;
    if (r < nrows) {
      const int nchunk = H / (8 * geo.wpr);  // uint4 chunks of this warp's part of the row
      const uint4* wrow = reinterpret_cast<const uint4*>(wrs + (size_t)r * H) + part * nchunk;
#pragma unroll 2
      for (int i = lane; i < nchunk; i += 32) {
        const uint4 wv = wrow[i];
#pragma unroll
        for (int t = 0; t < kNarrowT; ++t) {
          if (t < T) {
            const uint4 xv = reinterpret_cast<const uint4*>(xraw + (size_t)t * H)[part * nchunk + i];
            acc[t] += dot8_bf16(wv, xv);
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kNarrowT; ++t) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xFFFFFFFFu, acc[t], off);
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < kNarrowT; ++t) red[warp * kNarrowT + t] = acc[t];
    }
  }
  __syncthreads();
  if (tid < nrows * T) {
    const int rl = tid / T, t = tid % T;
    float s = red[(rl * geo.wpr) * kNarrowT + t];
    for (int p = 1; p < geo.wpr; ++p) s += red[(rl * geo.wpr + p) * kNarrowT + t];
    ws.logits[(size_t)t * E + row0 + rl] = s;
  }
  __syncthreads();
  if (tid == 0) grid_arrive(&ws.ctl[kCtlBar1]);

  // ---------------- activation operand of every token, in this CTA's shared memory
  if (warp < T) {
    float m = 0.0f;
    const uint32_t* xr = reinterpret_cast<const uint32_t*>(xraw + (size_t)warp * H);
    for (int i = lane; i < H / 2; i += 32) {
      const uint32_t v = xr[i];
      m = fmaxf(m, fmaxf(fabsf(bf16_lo(v)), fabsf(bf16_hi(v))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if (lane == 0) {
      shift_s[warp] = token_shift(m);
      xfac_s[warp] = mode == 0 ? pow2f(shift_s[warp]) : xS;
    }
  }
  __syncthreads();
  {
    const int nb = H / 16;
    for (int blk = tid; blk < T * nb; blk += kDcThreads) {
      const int t = blk / nb, bb = blk % nb;
      const uint4* src = reinterpret_cast<const uint4*>(xraw + (size_t)t * H + bb * 16);
      const uint4 u0 = src[0], u1 = src[1];
      const uint32_t words[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_lo(words[i]);
        v[2 * i + 1] = bf16_hi(words[i]);
      }
      __half hv[16];
      if (mode == 0) {
        const float f = pow2f(-shift_s[t]);
#pragma unroll
        for (int i = 0; i < 16; ++i) hv[i] = __float2half_rn(__fmul_rn(v[i], f));
      } else {
        uint32_t codes[2];
        const uint32_t sf = quantize16(v, xS, x_inv6S, codes);
        if (blk % G == b) {   // this CTA's share of the published W4A4 activation codes
          *reinterpret_cast<uint2*>(ws.xq + (size_t)t * (H / 2) + bb * 8) =
              make_uint2(codes[0], codes[1]);
          ws.xsf[(size_t)t * (H / 16) + bb] = static_cast<uint8_t>(sf);
        }
        const float sfv = e4m3_value_nonneg(sf);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          hv[i] = __float2half_rn(e2m1_value((codes[i >> 3] >> (4 * (i & 7))) & 0xF) * sfv);
      }
      // element 128J + 32c + 8p + q of the row is stored at 128J + 32p + 8c + q
      const int J = bb >> 3, c = (bb & 7) >> 1, p0 = 2 * (bb & 1);
      unsigned char* row = xop + (size_t)t * geo.x_stride + (size_t)(J * 128 + 8 * c) * 2;
      *reinterpret_cast<uint4*>(row + 64 * p0) = *reinterpret_cast<uint4*>(&hv[0]);
      *reinterpret_cast<uint4*>(row + 64 * (p0 + 1)) = *reinterpret_cast<uint4*>(&hv[8]);
    }
  }
  if (tid == 0 && !grid_wait(&ws.ctl[kCtlBar1], (uint32_t)G)) {
    record_status(ws.ctl, kStTimeout);
    abort_s = 1;
  }
  __syncthreads();
  __threadfence();

  // ---------------- 2. routing, in every CTA
  int32_t* cnt = reinterpret_cast<int32_t*>(arena);          // [E+1] counts -> offsets
  int32_t* uq = cnt + (E + 1);                               // [E+1] distinct -> group ids
  uint32_t* tmask = reinterpret_cast<uint32_t*>(uq + (E + 1));   // [E] tokens per expert
  for (int e = tid; e <= E; e += kDcThreads) {
    cnt[e] = 0;
    uq[e] = 0;
    if (e < E) tmask[e] = 0u;
  }
  if (warp < T) {
    int e_sel;
    float w_sel;
    topk_row(ws.logits + (size_t)warp * E, E, k, lane, e_sel, w_sel);
    if (lane < k) {
      sel_idx[warp * k + lane] = e_sel;
      sel_w[warp * k + lane] = w_sel;
    }
  }
  __syncthreads();
  if (tid < S) {
    atomicAdd(&cnt[sel_idx[tid]], 1);
    atomicOr(&tmask[sel_idx[tid]], 1u << (tid / k));
  }
  __syncthreads();
  for (int e = tid; e < E; e += kDcThreads) uq[e] = cnt[e] > 0 ? 1 : 0;
  __syncthreads();
  if (warp == 0) {
    warp_exclusive_scan(cnt, E, lane);
  } else if (warp == 1) {
    const int U = warp_exclusive_scan(uq, E, lane);
    if (lane == 0) U_s = U;
  }
  __syncthreads();
  for (int e = tid; e < E; e += kDcThreads) {
    const uint32_t tm = tmask[e];
    if (tm) {
      DcGroup gr;
      gr.expert = e;
      gr.slot0 = cnt[e];
      gr.n = __popc(tm);
      uint32_t toks = 0, mm = tm;
      for (int r = 0; mm; ++r) {
        const int t = __ffs(mm) - 1;
        toks |= (uint32_t)t << (4 * r);
        mm &= mm - 1;
      }
      gr.toks = toks;
      gr.mg = __ldg(&pk.mult[e * 3 + 0]);
      gr.mu = __ldg(&pk.mult[e * 3 + 1]);
      gr.md = __ldg(&pk.mult[e * 3 + 2]);
      gr.sd = __ldg(&pk.down_in_scale[e]);
      gr.i6d = __ldg(&pk.down_inv6S[e]);
      gr.pad[0] = gr.pad[1] = gr.pad[2] = 0;
      grp[uq[e]] = gr;
    }
  }
  if (tid < S) {
    // a token selects an expert at most once: its rank among the expert's slots is the
    // number of earlier tokens that selected the same expert
    const int t = tid / k, e = sel_idx[tid];
    sel_slot[tid] = cnt[e] + __popc(tmask[e] & ((1u << t) - 1u));
  }
  __syncthreads();
  const int U = U_s;
  if (b == 0) {
    for (int e = tid; e < E; e += kDcThreads) {
      ws.counts[e] = __popc(tmask[e]);
      ws.offsets[e] = cnt[e];
    }
    if (tid < S) {
      ws.idx[tid] = sel_idx[tid];
      ws.w[tid] = sel_w[tid];
      ws.slot_of[tid] = sel_slot[tid];
      ws.perm[sel_slot[tid]] = tid / k;
    }
    if (tid == 0) {
      ws.offsets[E] = S;
      ws.ctl[kCtlGroups] = (uint32_t)U;
      ws.ctl[kCtlUnique] = (uint32_t)U;
    }
  }
  __syncthreads();   // the routing scratch in the arena is dead from here on

  const int gu_tiles = I / 16, dn_tiles = H / kDnRows;
  int q0, q1, d0, d1;
  balanced_range(U * gu_tiles, q0, q1);
  balanced_range(U * dn_tiles, d0, d1);

  if (warp == kDcWarps) {
    // ---------------- producer: gate/up tasks, then this CTA's down tasks
    if (lane != 0) return;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t half = geo.row_bytes;
    int chunk = 0;
    for (int q = q0; q < q1 && !abort_s; ++q) {
      const int gi = q / gu_tiles, it = q % gu_tiles;
      const int e = grp[gi].expert;
      const size_t grow0 = (size_t)e * I + (size_t)it * 16;
      const uint8_t* gsrc = pk.gate_codes + grow0 * (H / 2);
      const uint8_t* usrc = pk.up_codes + grow0 * (H / 2);
      const uint8_t* gsc = pk.gu_scales + (((size_t)0 * pk.E + e) * gu_tiles + it) * (size_t)H;
      const uint8_t* usc = pk.gu_scales + (((size_t)1 * pk.E + e) * gu_tiles + it) * (size_t)H;
      for (int kc = 0; kc < geo.nkc; ++kc, ++chunk) {
        const int s = chunk % geo.gu_stages, n = chunk / geo.gu_stages;
        if (n > 0 && !mbar_wait(&gempty[s], (n - 1) & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
          break;
        }
        unsigned char* st = arena + (size_t)s * geo.gu_stage;
        mbar_arrive_expect_tx(&gfull[s], 32 * half + 2 * geo.KC);
        if (geo.nkc == 1) {
          bulk_g2s(st, gsrc, 16 * half, &gfull[s]);
          bulk_g2s(st + 16 * half, usrc, 16 * half, &gfull[s]);
        } else {
          for (int r = 0; r < 16; ++r) {
            bulk_g2s(st + r * half, gsrc + (size_t)r * (H / 2) + (size_t)kc * half, half,
                     &gfull[s]);
            bulk_g2s(st + (16 + r) * half, usrc + (size_t)r * (H / 2) + (size_t)kc * half, half,
                     &gfull[s]);
          }
        }
        bulk_g2s(st + 32 * half, gsc + (size_t)kc * geo.KC, geo.KC, &gfull[s]);
        bulk_g2s(st + 32 * half + geo.KC, usc + (size_t)kc * geo.KC, geo.KC, &gfull[s]);
      }
    }
    // the arena becomes the down ring once the consumers have released every gate/up stage
    const int used = chunk < geo.gu_stages ? chunk : geo.gu_stages;
    for (int i = 0; i < used && !abort_s; ++i) {
      const int c2 = chunk - 1 - i;
      if (!mbar_wait(&gempty[c2 % geo.gu_stages], (c2 / geo.gu_stages) & 1)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
      }
    }
    const uint32_t code_bytes = (uint32_t)kDnRows * (I / 2);
    int dchunk = 0;
    for (int q = d0; q < d1 && !abort_s; ++q, ++dchunk) {
      const int gi = q / dn_tiles, ht = q % dn_tiles;
      const int e = grp[gi].expert;
      const int s = dchunk % geo.dn_stages, n = dchunk / geo.dn_stages;
      if (n > 0 && !mbar_wait(&dempty[s], (n - 1) & 1)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
        break;
      }
      unsigned char* st = arena + (size_t)s * geo.dn_stage;
      mbar_arrive_expect_tx(&dfull[s], code_bytes + 8u * I);
      bulk_g2s(st, pk.down_codes + ((size_t)e * H + (size_t)ht * kDnRows) * (I / 2), code_bytes,
               &dfull[s]);
      bulk_g2s(st + code_bytes,
               pk.down_scales + ((size_t)e * (H / 64) + 2 * (size_t)ht) * (4 * (size_t)I), 8u * I,
               &dfull[s]);
    }
    // do not leave while copies into this CTA's shared memory may still be in flight
    const int dused = dchunk < geo.dn_stages ? dchunk : geo.dn_stages;
    for (int i = 0; i < dused; ++i) {
      const int c2 = dchunk - 1 - i;
      (void)mbar_wait(&dfull[c2 % geo.dn_stages], (c2 / geo.dn_stages) & 1);
    }
    return;
  }

  // ---------------- 3. gate/up + SiLU*up (consumer warps)
  const int g = lane >> 2, c = lane & 3;
  {
    int chunk = 0;
    const int jb_per_chunk = geo.KC / 128;
    for (int q = q0; q < q1; ++q) {
      const int gi = q / gu_tiles, it = q % gu_tiles;
      const DcGroup& gm = grp[gi];
      const int slot0 = gm.slot0, n = gm.n;
      const bool gvalid = g < n;
      const int xrow = gvalid ? group_tok(gm.toks, g) : 0;
      const unsigned char* xr = xop + (size_t)xrow * geo.x_stride + c * 16;
      float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kc = 0; kc < geo.nkc; ++kc, ++chunk) {
        const int s = chunk % geo.gu_stages, nn = chunk / geo.gu_stages;
        if (!abort_s && !mbar_wait(&gfull[s], nn & 1)) {
          record_status(ws.ctl, kStTimeout);
          abort_s = 1;
        }
        const unsigned char* st = arena + (size_t)s * geo.gu_stage;
        const unsigned char* scb = st + 32 * geo.row_bytes + c * 32 + g * 4;
        for (int jb = warp; jb < jb_per_chunk; jb += kDcWarps) {
          const int off = jb * 64 + c * 16;
          const uint4 gr = lds128(st + g * geo.row_bytes + off);
          const uint4 gr8 = lds128(st + (g + 8) * geo.row_bytes + off);
          const uint4 ur = lds128(st + (16 + g) * geo.row_bytes + off);
          const uint4 ur8 = lds128(st + (24 + g) * geo.row_bytes + off);
          const uint32_t scg = lds32(scb + jb * 128);
          const uint32_t scu = lds32(scb + geo.KC + jb * 128);
          uint4 xb[4];
          if (gvalid) {
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
        if (lane == 0) mbar_arrive(&gempty[s]);
      }
      // fixed-order reduction over the consumer warps
      float* myred = red + (size_t)(warp * 2) * 128;
      *reinterpret_cast<float4*>(myred + lane * 4) =
          make_float4(accg[0], accg[1], accg[2], accg[3]);
      *reinterpret_cast<float4*>(myred + 128 + lane * 4) =
          make_float4(accu[0], accu[1], accu[2], accu[3]);
      consumer_sync(kDcCons);
      if (warp == 0) {
        float G4[4] = {0.f, 0.f, 0.f, 0.f}, U4[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < kDcWarps; ++w) {
          const float4 a = *reinterpret_cast<const float4*>(red + (size_t)(w * 2) * 128 + lane * 4);
          const float4 bq =
              *reinterpret_cast<const float4*>(red + (size_t)(w * 2) * 128 + 128 + lane * 4);
          G4[0] += a.x; G4[1] += a.y; G4[2] += a.z; G4[3] += a.w;
          U4[0] += bq.x; U4[1] += bq.y; U4[2] += bq.z; U4[3] += bq.w;
        }
        float hv[4];  // (row g, col 2c), (row g, col 2c+1), (row g+8, col 2c), (row g+8, col 2c+1)
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
          const int col = 2 * c + (q2 & 1);
          const float xf = col < n ? xfac_s[group_tok(gm.toks, col)] : 0.0f;
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
            for (int off = 4; off < 32; off <<= 1)
              a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
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
            for (int off = 4; off < 32; off <<= 1)
              a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
            const uint32_t sf = e4m3_encode_rn(__fmul_rn(a, i6));
            uint32_t lo = 0, hi = 0;
            if (sf != 0u) {
              const float r = __frcp_rn(__fmul_rn(e4m3_value_nonneg(sf), Sd));
              lo = e2m1_encode_rn(__fmul_rn(v_lo, r)) << (4 * g);
              hi = e2m1_encode_rn(__fmul_rn(v_hi, r)) << (4 * g);
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
      consumer_sync(kDcCons);
    }
  }

  // ---------------- barrier 2: every CTA's h is written
  if (tid == 0) {
    grid_arrive(&ws.ctl[kCtlBar2]);
    if (!grid_wait(&ws.ctl[kCtlBar2], (uint32_t)G)) {
      record_status(ws.ctl, kStTimeout);
      abort_s = 1;
    }
    __threadfence();
  }
  consumer_sync(kDcCons);

  // ---------------- 4. down + combine (consumer warps)
  {
    const int nkb = I / 64;
    const uint32_t code_bytes = (uint32_t)kDnRows * (I / 2);
    int cur = -1, dchunk = 0;
    for (int q = d0; q < d1; ++q, ++dchunk) {
      const int gi = q / dn_tiles, ht = q % dn_tiles;
      const DcGroup& gm = grp[gi];
      const int slot0 = gm.slot0, n = gm.n;
      if (gi != cur) {
        // the group's h rows as the f16 operand: BF16 h * 2^-s (W4A16; s from the slot's
        // amax, exact), or the decoded NVFP4 code * scale (W4A4, exact)
        consumer_sync(kDcCons);
        if (tid < n) {
          if (mode == 0) {
            const int sh = amax_shift(__uint_as_float(__ldcg(&ws.slot_amax[slot0 + tid])));
            hfac_s[tid] = pow2f(sh);
            hinv_s[tid] = pow2f(-sh);
          } else {
            hfac_s[tid] = gm.sd;
          }
        }
        consumer_sync(kDcCons);
        const int words = n * (I / 2);
        for (int i0 = tid; i0 < words; i0 += 4 * kDcCons) {
          uint32_t v[4], sc[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kDcCons;
            const int row = i / (I / 2), wd = i % (I / 2);
            v[u] = 0u;
            sc[u] = 0u;
            if (i < words) {
              if (mode == 0) {
                v[u] = __ldcg(reinterpret_cast<const unsigned int*>(ws.h16 +
                                                                   (size_t)(slot0 + row) * I) + wd);
              } else {
                v[u] = __ldcg(ws.hq + (size_t)(slot0 + row) * (I / 2) + wd);
                sc[u] = __ldcg(ws.hsf + (size_t)(slot0 + row) * (I / 16) + wd / 8);
              }
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kDcCons;
            if (i < words) {
              const int row = i / (I / 2), wd = i % (I / 2);
              unsigned char* dst = xop + (size_t)row * geo.h_stride + wd * 4;
              if (mode == 0) {
                const float f = hinv_s[row];
                *reinterpret_cast<__half2*>(dst) =
                    __floats2half2_rn(__fmul_rn(__uint_as_float(v[u] << 16), f),
                                      __fmul_rn(__uint_as_float(v[u] & 0xFFFF0000u), f));
              } else {
                const float sv = e4m3_value_nonneg(sc[u]);
                *reinterpret_cast<__half2*>(dst) = __floats2half2_rn(
                    e2m1_value(v[u] & 0xF) * sv, e2m1_value((v[u] >> 4) & 0xF) * sv);
              }
            }
          }
        }
        consumer_sync(kDcCons);
        cur = gi;
      }
      const int s = dchunk % geo.dn_stages, nn = dchunk / geo.dn_stages;
      if (!abort_s && !mbar_wait(&dfull[s], nn & 1)) {
        record_status(ws.ctl, kStTimeout);
        abort_s = 1;
      }
      const unsigned char* st = arena + (size_t)s * geo.dn_stage;
      const bool gvalid = g < n;
      const unsigned char* hr = xop + (size_t)(gvalid ? g : 0) * geo.h_stride + c * 32;
      const unsigned char* rg = st + (size_t)(warp * 16 + g) * (I / 2) + c * 8;
      const unsigned char* rg8 = rg + 8 * (I / 2);
      const unsigned char* scb = st + code_bytes + (size_t)(warp >> 2) * (4 * I) +
                                 (size_t)(warp & 3) * nkb * 64 + c * 16 + g * 2;
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
      if (lane == 0) mbar_arrive(&dempty[s]);
      const float md = gm.md;
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        const int col = 2 * c + (q2 & 1);
        if (col < n) {
          const float y = acc[q2] * md * hfac_s[col];
          const int row = ht * kDnRows + warp * 16 + g + ((q2 >> 1) << 3);
          ws.y[(size_t)(slot0 + col) * H + row] = f32_to_bf16_rn(y);
        }
      }
      // the last task of output tile ht (one per group) forms out for its rows
      consumer_sync(kDcCons);
      if (tid == 0) {
        __threadfence();
        last_s = atomicAdd(&ws.ctl[kCtlTiles + ht], 1u) == (uint32_t)(U - 1) ? 1 : 0;
        __threadfence();
      }
      consumer_sync(kDcCons);
      if (last_s) {
        for (int it2 = tid; it2 < T * (kDnRows / 8); it2 += kDcCons) {
          const int t = it2 / (kDnRows / 8), r8 = ht * (kDnRows / 8) + it2 % (kDnRows / 8);
          float acc8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          for (int j0 = 0; j0 < k; j0 += 8) {
            float wj[8];
            int sj[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const bool ok = j0 + u < k;
              wj[u] = ok ? sel_w[t * k + j0 + u] : 0.0f;
              sj[u] = ok ? sel_slot[t * k + j0 + u] : -1;
            }
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
              v[u] = sj[u] >= 0 ? __ldcg(reinterpret_cast<const uint4*>(ws.y + (size_t)sj[u] * H) + r8)
                                : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              if (sj[u] < 0) break;
              const uint32_t wd[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
              for (int z = 0; z < 4; ++z) {
                acc8[2 * z] += wj[u] * __uint_as_float(wd[z] << 16);
                acc8[2 * z + 1] += wj[u] * __uint_as_float(wd[z] & 0xFFFF0000u);
              }
            }
          }
          uint32_t o[4];
#pragma unroll
          for (int z = 0; z < 4; ++z)
            o[z] = (uint32_t)f32_to_bf16_rn(acc8[2 * z]) |
                   ((uint32_t)f32_to_bf16_rn(acc8[2 * z + 1]) << 16);
          reinterpret_cast<uint4*>(out + (size_t)t * H)[r8] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }

  // ---------------- the last CTA to finish resets the kernel's control words
  consumer_sync(kDcCons);
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&ws.ctl[kCtlDone], 1u) == (uint32_t)(G - 1)) {
      ws.ctl[kCtlBar1] = 0u;
      ws.ctl[kCtlBar2] = 0u;
      for (int i = 0; i < dn_tiles; ++i) ws.ctl[kCtlTiles + i] = 0u;
      ws.ctl[kCtlDone] = 0u;
    }
  }
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl(const LaunchCfg& lc, Kern kern, dim3 grid, dim3 block, size_t smem,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = lc.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

// Geometry of the fused kernel for a shape, or false when it does not fit one SM's shared
// memory (the multi-kernel path serves such shapes).
bool decode_geom(int T, int H, int E, int k, int I, int num_ctas, void* out_geom) {
  DcGeom g{};
  if (T < 1 || T > kNarrowT || num_ctas < 1 || H / kDnRows > kCtlWords - kCtlTiles) return false;
  g.rows_max = (E + num_ctas - 1) / num_ctas;
  if (g.rows_max > kDcWarps) return false;
  g.wpr = g.rows_max <= kDcWarps / 2 ? 2 : 1;
  g.KC = H <= 4096 ? H : 4096;
  while (H % g.KC) g.KC -= 128;
  g.nkc = H / g.KC;
  g.row_bytes = g.KC / 2;
  g.gu_stage = 32 * g.row_bytes + 2 * g.KC;
  g.dn_stage = kDnRows * (I / 2) + 8 * I;
  g.x_stride = 2 * H + 64;
  g.h_stride = 2 * I + 16;
  g.xop = T * g.x_stride > kGroup * g.h_stride ? T * g.x_stride : kGroup * g.h_stride;
  g.smax = T * k;
  g.gmax = g.smax < E ? g.smax : E;
  const int route_bytes = g.rows_max * H * 2 + T * H * 2;
  const int scratch = (3 * E + 2) * 4;
  const int fixed = g.xop + kDcWarps * 2 * 128 * 4 + g.gmax * (int)sizeof(DcGroup) +
                    g.smax * 12 + 8 + 8 * (2 * 3 + 2 * 16 + 2) + kDcStatic;
  const int avail = kDcSmemMax - fixed;
  g.gu_stages = avail / g.gu_stage;
  if (g.gu_stages > 3) g.gu_stages = 3;
  if (g.gu_stages < 1) return false;
  int arena = g.gu_stages * g.gu_stage;
  if (arena < route_bytes) arena = route_bytes;
  if (arena < scratch) arena = scratch;
  if (arena > avail) return false;
  g.dn_stages = arena / g.dn_stage;
  if (g.dn_stages > 16) g.dn_stages = 16;
  if (g.dn_stages < 1) return false;
  g.arena = (arena + 127) & ~127;
  g.smem = g.arena + fixed - kDcStatic;
  if (g.smem + kDcStatic > kDcSmemMax) return false;
  if (out_geom) *static_cast<DcGeom*>(out_geom) = g;
  return true;
}

size_t decode_geom_bytes() { return sizeof(DcGeom); }

cudaError_t launch_decode(const LaunchCfg& lc, const PackView& pk, const WsView& ws, int mode,
                          float xS, float x_inv6S, const uint16_t* x, const uint16_t* wr,
                          uint16_t* out) {
  DcGeom geo;
  if (!decode_geom(ws.T, ws.H, ws.E, ws.k, ws.I, lc.num_sms, &geo)) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(k_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, geo.smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(lc, k_decode, dim3(lc.num_sms), dim3(kDcThreads), (size_t)geo.smem, pk, ws,
                    geo, x, wr, mode, xS, x_inv6S, out);
}

}  // namespace moe
