// moe_internal.cuh — device helpers and views shared by the sm_103a kernels of the NVFP4
// routed-expert MoE library. Internal to the library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

// Device status codes (values equal the public moe_status codes).
constexpr uint32_t kStOk = 0;
constexpr uint32_t kStTimeout = 5;

// A wait that takes longer than this gives up, records kStTimeout and returns.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Narrow (decode) path: tokens per call at most this many; also the token-group width of the
// grouped path (the N of one m16n8k16 MMA).
constexpr int kNarrowT = 8;
constexpr int kGroup = 8;
// The fused narrow kernel writes its tagged logits this many times ([replica][T][E]); CTA b
// polls replica b % kLogitReplicas, which spreads the 152 readers over more L2 lines.
constexpr int kLogitReplicas = 8;

// ------------------------------------------------------------------ workspace view
// Control words at the start of the workspace (zero-filled before first use).
enum : int {
  kCtlRouteTicket = 0,  // last-block-done ticket of the narrow router (self-resetting)
  kCtlStatus = 1,       // first device error (sticky until read by the host)
  kCtlGroups = 2,       // number of token groups of the current call
  kCtlUnique = 3,       // number of distinct experts of the current call
  kCtlTokenTiles = 4,   // number of 128-slot token tiles (grouped tensor-core path)
  kCtlEpoch = 8,        // fused narrow kernel: epoch of the last completed call (tags its data)
  kCtlDone = 9,         //   CTAs finished, over all calls (the last of a call advances the epoch)
  kCtlXShare = 10,      //   CTAs that published their share of the quantised activations, over
                        //   all calls ((epoch - 1) * CTAs at the start of a call)
  kCtlWords = 64
};

// Per token group (<= 8 tokens of one expert): everything the expert kernels need about it,
// written by the routing stage so that the expert kernels stage it with one load.
struct GroupMeta {
  int32_t expert, slot0, n, pad0;
  int32_t tok[8];        // token ids of the group's columns (-1 past n)
  float mg, mu, md, sd;  // gate/up/down multipliers, down input scale
  float i6d, pad1, pad2, pad3;  // fl32(1/fl32(6*sd))
};
static_assert(sizeof(GroupMeta) == 80, "GroupMeta layout");

struct WsView {
  uint32_t* ctl;
  GroupMeta* gmeta;    // [G]
  uint32_t* slot_amax; // [T*k] bits of max|h| per slot (W4A16), zeroed by the routing stage
  float* logits;       // [T][E] (fused narrow kernel: [replica][T][E] 64-bit {logit, epoch})
  int32_t* idx;        // [T][k]
  float* w;            // [T][k]
  int32_t* slot_of;    // [T][k]
  int32_t* counts;     // [E]
  int32_t* offsets;    // [E+1]
  int32_t* perm;       // [T*k]
  int32_t* chunk_base; // [nchunk][E] (grouped routing)
  __half* xh;          // [T][H] activations as the f16 B operand of gate/up
  float* xfac;         // [T] factor restoring xh's scale (2^shift in W4A16, S_x in W4A4)
  uint8_t* xq;         // [T][H/2]  W4A4 activation codes ([T][H] E4M3 codes in W4A8)
  uint8_t* xsf;        // [T][H/16] W4A4 activation scales
  uint16_t* h16;       // [T*k][I] W4A16 h (BF16)
  uint8_t* hq;         // [T*k][I/2] W4A4 h codes ([T*k][I] E4M3 codes in W4A8)
  uint8_t* hsf;        // [T*k][I/16] W4A4 h scales
  uint16_t* y;         // [T*k][H] BF16 expert outputs
  // fused narrow kernel: 64-bit words {data, epoch} that other CTAs poll instead of a barrier
  unsigned long long* htag;  // [T*k][I/16][9]: h of one 16-element block (W4A16: 8 BF16 pairs +
                             // max |h|; W4A4: code words lo, hi + scale byte)
  unsigned long long* ytag;  // [T*k][H/2]: BF16 pairs of Y
  // grouped tensor-core path: token tiles of <= 128 slots of one expert; tile j occupies padded
  // rows ("pslots") 128j .. 128j+127 of the permuted operands
  int32_t* tt_expert;  // [NT]
  int32_t* tt_slot0;   // [NT] first (unpadded) slot of the tile
  int32_t* tt_n;       // [NT] slots in the tile (1..128)
  int32_t* ttbase;     // [E+1] first token tile of each expert
  uint8_t* xq_perm;    // [128*NT][H/2]  activation codes by pslot (W4A4)
  uint8_t* xsf_atoms;  // [NT][H/64][512] activation scales in tensor-core scale-factor atoms
  uint8_t* hq_perm;    // [128*NT][I/2]  h codes by pslot
  uint8_t* hsf_atoms;  // [NT][I/64][512]
  __half* xh_perm;     // W4A16 grouped path: [128*NT][H] f16(x * 2^-s) by pslot
  __half* hf_perm;     // W4A16 grouped path: [128*NT][I] f16(h * 2^-s) by pslot
  // shared expert (null when the call has none): its FP32 output before the BF16 rounding and
  // its gate, read by the combines
  const float* sh_y;      // [T][H]
  const float* sh_sigma;  // [T]
  // narrow calls with the shared expert inside the fused kernel: tagged words of its h
  // ([T][Is]), its gate ([T]) and its output Ys ([T][H]), in that order
  unsigned long long* sh_tag;
  int T, H, E, k, I, G, NT;
};

// Moves a (non-null) workspace pointer by `off` bytes: the regions of a stack's layers.
template <typename P>
__host__ __device__ __forceinline__ void shift_ptr(P*& p, size_t off) {
  if (p) p = reinterpret_cast<P*>(reinterpret_cast<unsigned char*>(p) + off);
}

// The shared expert of a call: caller-owned BF16 weights and workspace buffers.
struct ShView {
  const uint16_t* gate_up;  // [2 Is][H]: gate rows, then up rows
  const uint16_t* down;     // [H][Is]
  const uint16_t* gate;     // [H] gate vector
  uint16_t* hs;             // [T][Is] BF16 h
  float* sigma;             // [T]
  float* ys;                // [T][H] FP32
  float* gu;                // [T][2 Is] FP32 gate/up products (wide calls)
  int Is;
};

// ------------------------------------------------------------------ pack view
// Codes keep the checkpoint layout ([rows][cols/2] per matrix, experts contiguous).
// Scales are stored in the "fragment" order the narrow/grouped kernels read:
//   gate/up: [mat(2)][E][I/16 row tiles][H/128 k-blocks][c(4)][g(8)][4]
//            bytes (c, g, 2h + b) of k-block J: the scale of row 16*tile + g + 8h, block 8J+2c+b.
//   down:    [E][H/64 row tiles][4 m16 tiles][I/64 k-blocks][c(4)][g(8)][2]
struct PackView {
  const uint8_t* gate_codes;   // [E][I][H/2]
  const uint8_t* up_codes;     // [E][I][H/2]
  const uint8_t* down_codes;   // [E][H][I/2]
  const uint8_t* gu_scales;    // see above
  const uint8_t* down_scales;  // see above
  const float* mult;           // [E][3]
  const float* down_in_scale;  // [E]
  const float* down_inv6S;     // [E] fl32(1 / fl32(6 * S_down))
  // tensor-core scale-factor atoms (512 B = 128 rows x 4 blocks of 16; byte
  // (r % 32) * 16 + (r / 32) * 4 + b), one per (row tile, K step of 64):
  //   sfa_gu:   [E][I/64][H/64]: the 64 gate and 64 up rows of intermediate tile mt interleaved
  //             by 16 (rows 32q .. 32q+15: gate rows 64*mt + 16q .., 32q+16 .. +31: the up rows)
  //   sfa_down: [E][H/128][I/64]
  const uint8_t* sfa_gu;
  const uint8_t* sfa_down;
  int E, H, I;
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase: false after limit_ns (kWaitLimitNs unless a kernel passes
// its own).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// One TMA bulk copy global -> shared (16-byte aligned, bytes % 16 == 0), completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void record_status(uint32_t* ctl, uint32_t code) {
  atomicCAS(&ctl[kCtlStatus], 0u, code);
}

// Programmatic dependent launch: wait for the preceding kernel's results / let the next
// kernel start its prologue.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ format conversions
// Four bytes of E2M1 codes -> four f16x2 (byte b -> out[b]; low nibble -> low half). Exact.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t src, uint32_t (&out)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}\n"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(src));
}

// Two E4M3 bytes (low byte -> low half) -> f16x2. Exact (every E4M3 value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t out;
  uint16_t in = static_cast<uint16_t>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(in));
  return out;
}

// a * (low half of s), a * (high half of s): the half broadcast is an operand selector of the
// f16x2 multiply, so two rows' scales share one conversion
__device__ __forceinline__ uint32_t hmul2_lo(uint32_t a, uint32_t s) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a),
                            __low2half2(*reinterpret_cast<const __half2*>(&s)));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hmul2_hi(uint32_t a, uint32_t s) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a),
                            __high2half2(*reinterpret_cast<const __half2*>(&s)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Exact decoded values.
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  const uint32_t e = (code >> 1) & 3u, m = code & 1u;
  // exponent field 0: 0 or 0.5; otherwise (1 + m/2) * 2^(e-1)
  const float v = (e == 0u) ? 0.5f * static_cast<float>(m) : __uint_as_float(((126u + e) << 23) | (m << 22));
  return (code & 8u) ? -v : v;
}

__device__ __forceinline__ float e4m3_value_nonneg(uint32_t byte) {
  uint32_t e = (byte >> 3) & 0xF, mnt = byte & 7;
  if (e == 0) return static_cast<float>(mnt) * 0.001953125f;  // m/8 * 2^-6
  return __uint_as_float(((e + 120u) << 23) | (mnt << 20));   // (1+m/8) * 2^(e-7)
}

// Round-to-nearest-even encoders of the quantiser, in exact integer/compare steps.
// E2M1: nearest of {0,.5,1,1.5,2,3,4,6}, ties to the even code, above 6 -> 6; sign kept.
__device__ __forceinline__ uint32_t e2m1_encode_rn(float v) {
  const float a = fabsf(v);
  uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
               (a >= 3.5f) + (a > 5.0f);
  return c | ((__float_as_uint(v) >> 28) & 8u);
}

// E4M3 of a non-negative finite float: nearest, ties to even, above 448 -> 448 (0x7E).
__device__ __forceinline__ uint32_t e4m3_encode_rn(float t) {
  if (!(t > 0.0f)) return 0u;
  if (t >= 448.0f) return 0x7Eu;
  if (t < 0.015625f) {  // subnormal range: multiples of 2^-9
    return static_cast<uint32_t>(__float2int_rn(t * 512.0f));  // 0..8 (8 == 2^-6, normal)
  }
  const uint32_t bits = __float_as_uint(t);
  const int e = static_cast<int>((bits >> 23) & 0xFF) - 127;   // t in [2^e, 2^(e+1))
  const float frac = __uint_as_float((bits & 0x7FFFFFu) | 0x3F800000u);  // in [1, 2)
  uint32_t m = static_cast<uint32_t>(__float2int_rn((frac - 1.0f) * 8.0f));
  uint32_t ef = static_cast<uint32_t>(e + 7);
  if (m == 8) { m = 0; ef += 1; }
  uint32_t r = (ef << 3) | m;
  return r > 0x7Eu ? 0x7Eu : r;
}

// W4A8 activation code: E4M3 of fl32(v * r8), nearest, ties to even, saturating at 448, with
// the sign of v kept (r8 = fl32(1 / fl32(6 S)) for the matrix's FP32 input scale S, which is the
// inv6S the packs hold; the decoded value is E4M3(code) * fl32(6 S)).
__device__ __forceinline__ uint32_t a8_encode(float v, float r8) {
  const float t = __fmul_rn(v, r8);
  return e4m3_encode_rn(fabsf(t)) | ((__float_as_uint(t) >> 24) & 0x80u);
}

// Quantise 16 FP32 values with per-matrix scale S (inv6S = fl32(1/fl32(6 S))).
// Writes 8 code bytes (even element in the low nibble) and returns the scale byte.
// Every step is one IEEE single-precision operation, as in the public quantiser definition.
__device__ __forceinline__ uint32_t quantize16(const float (&v)[16], float S, float inv6S,
                                               uint32_t (&codes)[2]) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(v[i]));
  const uint32_t sf = e4m3_encode_rn(__fmul_rn(a, inv6S));
  codes[0] = codes[1] = 0u;
  if (sf == 0u) return 0u;
  const float r = __frcp_rn(__fmul_rn(e4m3_value_nonneg(sf), S));
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t q = e2m1_encode_rn(__fmul_rn(v[i], r));
    codes[i >> 3] |= q << (4 * (i & 7));
  }
  return sf;
}

// ------------------------------------------------------------------ MMA
// D (16x8 f32) += A (16x16 f16, row) * B (16x8 f16, col).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The product of one 64-wide k-block for one m16 row tile and one 8-token group:
//   rowg / rowg8: the thread's 8 code bytes of rows g and g+8 (codes k = 64j+16c .. +15),
//   sc:           the two scale bytes (rows g, g+8) of block 4j + c,
//   xb0, xb1:     the thread's 16 B operand values x[g][64j+16c .. +15] as 2 x uint4.
// The k order inside an MMA is permuted consistently for A and B (thread c of MMA m holds
// k = 64j + 16c + 4m + {0,1,2,3}), so both operands come from contiguous bytes.
__device__ __forceinline__ void kblock_mma(float (&acc)[4], uint2 rowg, uint2 rowg8, uint32_t sc,
                                           const uint4& xb0, const uint4& xb1) {
  const uint32_t s01 = e4m3x2_to_f16x2(sc);   // {row g, row g+8}
  uint32_t ga[4], gb[4], ha[4], hb[4];
  e2m1x8_to_f16x2x4(rowg.x, ga);   // row g, k 0..7
  e2m1x8_to_f16x2x4(rowg.y, gb);   // row g, k 8..15
  e2m1x8_to_f16x2x4(rowg8.x, ha);  // row g+8
  e2m1x8_to_f16x2x4(rowg8.y, hb);
  const uint32_t xs[8] = {xb0.x, xb0.y, xb0.z, xb0.w, xb1.x, xb1.y, xb1.z, xb1.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t* g4 = (m < 2) ? ga : gb;
    const uint32_t* h4 = (m < 2) ? ha : hb;
    const int o = (m & 1) * 2;
    uint32_t a[4];
    a[0] = hmul2_lo(g4[o], s01);
    a[1] = hmul2_hi(h4[o], s01);
    a[2] = hmul2_lo(g4[o + 1], s01);
    a[3] = hmul2_hi(h4[o + 1], s01);
    mma_16816(acc, a, xs[2 * m], xs[2 * m + 1]);
  }
}

// The product of one 128-wide k-block for one m16 row tile and one 8-token group:
//   rowg / rowg8: the thread's 16 code bytes of rows g and g+8 (codes k = 128J + 32c .. +31),
//   sc4:          scale bytes (row g, block 2c), (row g, block 2c+1), (row g+8, 2c), (row g+8, 2c+1),
//   xb[p]:        the thread's B operand x[g][128J + 32c + 8p .. +7], p = 0..3.
// MMA m (0..7) holds k = 128J + 32c + 4m + {0,1,2,3}: the k order inside an MMA is permuted
// consistently for A and B so that each operand comes from contiguous bytes.
__device__ __forceinline__ void kblock128_mma(float (&acc)[4], const uint4& rowg, const uint4& rowg8,
                                              uint32_t sc4, const uint4 (&xb)[4]) {
  // {row g, row g+8} scales of block 2c and of block 2c+1
  const uint32_t s_0 = e4m3x2_to_f16x2(__byte_perm(sc4, 0u, 0x0020u));
  const uint32_t s_1 = e4m3x2_to_f16x2(__byte_perm(sc4, 0u, 0x0031u));
  const uint32_t gw[4] = {rowg.x, rowg.y, rowg.z, rowg.w};
  const uint32_t hw[4] = {rowg8.x, rowg8.y, rowg8.z, rowg8.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {   // word w = codes 8w..8w+7 -> MMAs 2w, 2w+1
    uint32_t gf[4], hf[4];
    e2m1x8_to_f16x2x4(gw[w], gf);
    e2m1x8_to_f16x2x4(hw[w], hf);
    const uint32_t sp = (w < 2) ? s_0 : s_1;
    const uint4& xv = xb[w];
    {
      uint32_t a[4] = {hmul2_lo(gf[0], sp), hmul2_hi(hf[0], sp), hmul2_lo(gf[1], sp),
                       hmul2_hi(hf[1], sp)};
      mma_16816(acc, a, xv.x, xv.y);
    }
    {
      uint32_t a[4] = {hmul2_lo(gf[2], sp), hmul2_hi(hf[2], sp), hmul2_lo(gf[3], sp),
                       hmul2_hi(hf[3], sp)};
      mma_16816(acc, a, xv.z, xv.w);
    }
  }
}

// ------------------------------------------------------------------ shared arithmetic helpers
// BF16 halves of a 32-bit word, the router dot product, the f16 operand's power-of-two
// scaling, the warp top-k, and small shared-memory / conversion helpers of the expert kernels.
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Sum of the 8 exact BF16 products of two uint4 chunks, as a fixed pairwise tree.
__device__ __forceinline__ float dot8_bf16(const uint4& a, const uint4& b) {
  const float p0 = bf16_lo(a.x) * bf16_lo(b.x), p1 = bf16_hi(a.x) * bf16_hi(b.x);
  const float p2 = bf16_lo(a.y) * bf16_lo(b.y), p3 = bf16_hi(a.y) * bf16_hi(b.y);
  const float p4 = bf16_lo(a.z) * bf16_lo(b.z), p5 = bf16_hi(a.z) * bf16_hi(b.z);
  const float p6 = bf16_lo(a.w) * bf16_lo(b.w), p7 = bf16_hi(a.w) * bf16_hi(b.w);
  return ((p0 + p1) + (p2 + p3)) + ((p4 + p5) + (p6 + p7));
}

// Power-of-two shift that puts a token's amax in [2^14, 2^15) for the f16 operand.
__device__ __forceinline__ int token_shift(float amax) {
  if (!(amax > 0.0f)) return 0;
  int e;
  frexpf(amax, &e);  // amax = f * 2^e, f in [0.5, 1)
  int s = e - 15;
  return s < -110 ? -110 : (s > 110 ? 110 : s);
}

__device__ __forceinline__ float pow2f(int s) { return __int_as_float((127 + s) << 23); }

// Orderable 32-bit key of an FP32 logit: a larger logit gives a larger key, and -0 and +0 give
// the same key. Key 0 lies below every logit and marks a taken or absent entry.
__device__ __forceinline__ uint32_t logit_key(float v) {
  uint32_t f = __float_as_uint(v);
  if (f == 0x80000000u) f = 0u;
  return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Top-k of one token's logits by one warp, followed by the softmax over the k selected logits.
// Lane e % 32 holds the key of logit e in key[e / 32] (0 for e >= E). Each round takes the
// warp's largest key (redux.sync max) and, among lanes holding it, the lowest expert index
// (redux.sync min): larger logit first, equal logits -> lower index first. The winning lane
// drops its entry; every lane rescans its registers (predicated, no divergent branch, which
// measured faster). Lane j < k returns the j-th selection and its softmax weight; the sum of
// exponentials is a fixed butterfly, identical in all lanes.
template <int V>
__device__ __forceinline__ void warp_select_softmax(uint32_t (&key)[V], int k, int lane,
                                                    int& e_out, float& w_out) {
  uint32_t bk = 0u;
  int bp = 0;
#pragma unroll
  for (int i = 0; i < V; ++i)
    if (key[i] > bk) { bk = key[i]; bp = i; }
  e_out = 0;
  float v = 0.0f;
  for (int j = 0; j < k; ++j) {
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, bk);
    const uint32_t ew =
        __reduce_min_sync(0xFFFFFFFFu, bk == m ? (uint32_t)(lane + 32 * bp) : 0xFFFFFFFFu);
    if (lane == j) {
      e_out = (int)ew;
      v = key_logit(m);
    }
    const int taken = (int)(ew & 31u) == lane ? bp : -1;
    uint32_t nb = 0u;
    int np = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      key[i] = i == taken ? 0u : key[i];
      if (key[i] > nb) { nb = key[i]; np = i; }
    }
    bk = nb;
    bp = np;
  }
  const float m0 = __shfl_sync(0xFFFFFFFFu, v, 0);
  const float ex = lane < k ? expf(v - m0) : 0.0f;
  float z = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, off);
  w_out = ex / z;
}

// Top-k + softmax of one token by one warp, with a 32-entry shared-memory scratch (cand):
// threshold L = the k-th largest of the 32 lane maxima (counted with multiplicity). The k lane
// maxima >= L are k distinct logits, so every one of the top k has key >= L. L is found without
// a sort: each lane counts the lane maxima above its own (broadcast reads of the 32 maxima from
// the scratch), and L is the smallest lane maximum with fewer than k above it. The candidates
// (keys >= L, about 12 of 512 for k = 10) are packed into the scratch by ballots, each
// candidate's exact rank by (key desc, index asc) is counted against the others, and ranks < k
// are the selection. More than 32 candidates: the redux.sync rounds of warp_select_softmax.
template <int V>
__device__ __forceinline__ void warp_select_scratch(uint32_t (&key)[V], int k, int lane,
                                                    unsigned long long* cand, int& e_out,
                                                    float& w_out) {
  static_assert((V & (V - 1)) == 0, "V is a power of two");
  uint32_t m[V];
#pragma unroll
  for (int i = 0; i < V; ++i) m[i] = key[i];
#pragma unroll
  for (int w = V / 2; w > 0; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = m[i] > m[i + w] ? m[i] : m[i + w];
  const uint32_t sv = m[0];
  uint32_t* lm = reinterpret_cast<uint32_t*>(cand);
  lm[lane] = sv;
  __syncwarp();
  int above = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 q = reinterpret_cast<const uint4*>(lm)[j];
    above += (q.x > sv) + (q.y > sv) + (q.z > sv) + (q.w > sv);
  }
  uint32_t thr = __reduce_min_sync(0xFFFFFFFFu, above < k ? sv : 0xFFFFFFFFu);
  if (thr == 0u) thr = 1u;   // fewer than k lanes hold logits: every logit is a candidate
  __syncwarp();              // every lane has read the maxima before the scratch is reused
  const unsigned lt = (1u << lane) - 1u;
  int C = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const bool is = key[i] >= thr;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, is);
    const int pos = C + __popc(bal & lt);
    // candidate word: key in the high half, ~index in the low half, so that a larger word is a
    // larger logit, and for equal logits the lower index
    if (is && pos < 32) cand[pos] = ((unsigned long long)key[i] << 32) | (uint32_t)~(lane + 32 * i);
    C += __popc(bal);
  }
  if (C > 32) {
    warp_select_softmax<V>(key, k, lane, e_out, w_out);
    return;
  }
  __syncwarp();
  e_out = 0;
  float v = 0.0f;
  int r = 32;
  unsigned long long mine = 0ull;
  if (lane < C) {
    mine = cand[lane];
    r = 0;
#pragma unroll 4
    for (int j = 0; j < (C + 1) >> 1; ++j) {   // broadcast reads; entries >= C do not count
      const ulonglong2 q = reinterpret_cast<const ulonglong2*>(cand)[j];
      r += (q.x > mine) + (2 * j + 1 < C && q.y > mine);
    }
  }
  __syncwarp();
  if (r < k) cand[r] = mine;   // cand[0..k) <- the selection in order
  __syncwarp();
  if (lane < k) {
    const unsigned long long w = cand[lane];
    e_out = (int)~(uint32_t)w;
    v = key_logit((uint32_t)(w >> 32));
  }
  __syncwarp();
  const float m0 = __shfl_sync(0xFFFFFFFFu, v, 0);
  const float ex = lane < k ? expf(v - m0) : 0.0f;
  float z = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, off);
  w_out = ex / z;
}

// The same for E <= 32 V FP32 logits in global memory (read through L2), with the shared-memory
// scratch selection above (cand: 32 words of this warp's shared memory).
template <int V>
__device__ __forceinline__ void warp_topk_softmax_scratch(const float* row, int E, int k, int lane,
                                                          unsigned long long* cand, int& e_out,
                                                          float& w_out) {
  uint32_t key[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? logit_key(__ldcg(row + e)) : 0u;
  }
  warp_select_scratch<V>(key, k, lane, cand, e_out, w_out);
}

__device__ __forceinline__ void topk_row_scratch(const float* row, int E, int k, int lane,
                                                 unsigned long long* cand, int& e_out,
                                                 float& w_out) {
  if (E <= 128) warp_topk_softmax_scratch<4>(row, E, k, lane, cand, e_out, w_out);
  else if (E <= 256) warp_topk_softmax_scratch<8>(row, E, k, lane, cand, e_out, w_out);
  else if (E <= 512) warp_topk_softmax_scratch<16>(row, E, k, lane, cand, e_out, w_out);
  else warp_topk_softmax_scratch<32>(row, E, k, lane, cand, e_out, w_out);
}

// The same for E <= 32 V FP32 logits in global memory (read through L2).
template <int V>
__device__ __forceinline__ void warp_topk_softmax(const float* row, int E, int k, int lane,
                                                  int& e_out, float& w_out) {
  uint32_t key[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? logit_key(__ldcg(row + e)) : 0u;
  }
  warp_select_softmax<V>(key, k, lane, e_out, w_out);
}

__device__ __forceinline__ void topk_row(const float* row, int E, int k, int lane, int& e_out,
                                         float& w_out) {
  if (E <= 128) warp_topk_softmax<4>(row, E, k, lane, e_out, w_out);
  else if (E <= 256) warp_topk_softmax<8>(row, E, k, lane, e_out, w_out);
  else if (E <= 512) warp_topk_softmax<16>(row, E, k, lane, e_out, w_out);
  else warp_topk_softmax<32>(row, E, k, lane, e_out, w_out);
}

__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

__device__ __forceinline__ uint2 lds64(const unsigned char* p) {
  return *reinterpret_cast<const uint2*>(p);
}
__device__ __forceinline__ uint4 lds128(const unsigned char* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ uint32_t lds16(const unsigned char* p) {
  return *reinterpret_cast<const uint16_t*>(p);
}
__device__ __forceinline__ uint32_t lds32(const unsigned char* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return (g / (1.0f + expf(-g))) * u;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

// v rounded to the nearest BF16 value (ties to even), as an FP32 value
__device__ __forceinline__ float bf16_round(float v) {
  return __uint_as_float((uint32_t)f32_to_bf16_rn(v) << 16);
}

__device__ __forceinline__ int amax_shift(float m) {
  if (!(m > 0.0f)) return 0;
  int ex;
  frexpf(m, &ex);
  const int sh = ex - 15;
  return sh < -110 ? -110 : (sh > 110 ? 110 : sh);
}

// ------------------------------------------------------------------ launchers
struct LaunchCfg {
  cudaStream_t stream;
  int num_sms;
  bool pdl;
};

// Per-launch profiling (measurement only): while `count` > 0 on this host thread, the i-th
// kernel launch of a call records ev[2i] before it and ev[2i+1] after it on the call's stream,
// and its function is kept in func[i]. Defined in moe_api.cu.
struct LaunchProf {
  cudaEvent_t ev[64];
  int count;            // events supplied (0: profiling off)
  int next;             // launches seen so far in the profiled call
  const void* func[32];
};
LaunchProf& launch_prof();

// Every kernel of a forward call is launched here: programmatic dependent launch when lc.pdl,
// and the profiling events above when they are active.
template <typename Kern, typename... Args>
cudaError_t launch_kernel(const LaunchCfg& lc, Kern kern, dim3 grid, dim3 block, size_t smem,
                          Args... args) {
  LaunchProf& prof = launch_prof();
  const int i = prof.next;
  const bool rec = 2 * i + 1 < prof.count;
  if (rec) {
    const cudaError_t e = cudaEventRecord(prof.ev[2 * i], lc.stream);
    if (e != cudaSuccess) return e;
  }
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (rec) {
    if (e == cudaSuccess) e = cudaEventRecord(prof.ev[2 * i + 1], lc.stream);
    if (i < 32) prof.func[i] = reinterpret_cast<const void*>(kern);
  }
  if (prof.count > 0) prof.next = i + 1;
  return e;
}

cudaError_t launch_route_narrow(const LaunchCfg& lc, const uint16_t* x, const uint16_t* wr,
                                const WsView& ws, const PackView* pk, int mode, float xS,
                                float x_inv6S,
                                int32_t* out_idx, float* out_w, int32_t* out_counts,
                                int32_t* out_offsets, int32_t* out_perm);
cudaError_t launch_route_wide(const LaunchCfg& lc, const uint16_t* x, const uint16_t* wr,
                              const WsView& ws, const PackView* pk, int32_t* out_idx, float* out_w,
                              int32_t* out_counts, int32_t* out_offsets, int32_t* out_perm,
                              int* launches);
cudaError_t launch_xprep_wide(const LaunchCfg& lc, const uint16_t* x, const WsView& ws, int mode,
                              float xS, float x_inv6S);
cudaError_t launch_quantize_rows(const LaunchCfg& lc, const uint16_t* x, int rows, int cols,
                                 float S, float inv6S, uint8_t* codes, uint8_t* scales);
cudaError_t launch_gateup(const LaunchCfg& lc, const PackView& pk, const WsView& ws, int mode,
                          bool x_resident);
cudaError_t launch_down(const LaunchCfg& lc, const PackView& pk, const WsView& ws, int mode,
                        bool h_resident);
cudaError_t launch_combine(const LaunchCfg& lc, const WsView& ws, uint16_t* out);
// Fused narrow-call kernel (router .. combine in one launch): whether a shape fits it, and the
// launch.
bool decode_geom(int T, int H, int E, int k, int I, int num_ctas, void* out_geom);
// xnext (or null): [T][H] receives BF16(x + out), the input of the next layer of a chained stack.
// sv (or null): the shared expert, computed inside the kernel (one or two tokens; the
// workspace's sh_tag words and sv's hs / sigma / ys receive its intermediates).
// cudaErrorNotSupported when it cannot be fused for the shape (the caller runs it separately).
cudaError_t launch_decode(const LaunchCfg& lc, const PackView& pk, const WsView& ws, int mode,
                          float xS, float x_inv6S, const uint16_t* x, const uint16_t* wr,
                          uint16_t* out, uint16_t* xnext, const ShView* sv = nullptr);
// out[i] = BF16(a[i] + b[i]) over n BF16 values (n % 8 == 0): a chained layer's next input.
cudaError_t launch_residual_add(const LaunchCfg& lc, const uint16_t* a, const uint16_t* b,
                                uint16_t* out, size_t n);
cudaError_t launch_pack_scales(cudaStream_t s, const uint8_t* raw_gate, const uint8_t* raw_up,
                               const uint8_t* raw_down, int E, int H, int I, uint8_t* gu_scales,
                               uint8_t* down_scales, uint8_t* sfa_gu, uint8_t* sfa_down);
// Grouped tensor-core experts (W4A4, wide calls): activation permutation, gate/up, down.
bool tc_supported();
// W4A4 grouped experts on tcgen05: activation quantisation + permutation, gate/up, down.
cudaError_t launch_tc_experts(const LaunchCfg& lc, const PackView& pk, const WsView& ws,
                              const uint16_t* x, float xS, float x_inv6S);
// W4A16 grouped experts on tcgen05 kind::f16 (weights dequantised in shared memory).
// a8 = 1: W4A8 (E4M3 activations with the scale fl32(6 xS), r8 = fl32(1/fl32(6 xS))).
cudaError_t launch_tc16_experts(const LaunchCfg& lc, const PackView& pk, const WsView& ws,
                                const uint16_t* x, int a8, float xS, float x_r8);
// Whether a wide call runs the tensor-core grouped path (128-slot token tiles) for its mode.
bool tile_path(int T, int H, int I, int mode);
// Router logits of a wide call on tcgen05 (BF16 x BF16 -> FP32).
cudaError_t launch_tc_router(const LaunchCfg& lc, const uint16_t* x, const uint16_t* wr,
                             const WsView& ws);
cudaError_t launch_unpack_scales(cudaStream_t s, const uint8_t* gu_scales,
                                 const uint8_t* down_scales, int E, int H, int I, int expert,
                                 int which, uint8_t* raw_out);

// The shared expert (BF16 SwiGLU with a sigmoid gate): h, the gate and the FP32 output for the
// combine; narrow calls on CUDA-core GEMVs, wide calls on the tcgen05 BF16 GEMM.
cudaError_t launch_shared(const LaunchCfg& lc, const uint16_t* x, const ShView& sv,
                          const WsView& ws, int* launches);

// Test-only fault injection (host side; see moe_test_inject_faults in the C ABI): the fused
// narrow-call kernel's wait bound and a CTA that publishes no logits, and device allocations of
// moe_pack_nvfp4 that fail.
struct FaultInjection {
  uint64_t wait_ns;        // 0: the default bound kWaitLimitNs
  int skip_logits_cta;     // -1: none
  int fail_pack_allocs;    // the next this many allocations of moe_pack_nvfp4 fail
};
FaultInjection& fault_injection();

// Dynamic shared memory the expert kernels need (host side, for validation).
size_t gateup_smem_bytes(int H, bool x_resident, int T);
size_t down_smem_bytes(int I, bool h_resident, int slots);

}  // namespace moe
