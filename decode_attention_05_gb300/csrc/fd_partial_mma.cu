// fd_partial_mma.cu -- split-KV partial pass with the GQA group's dot products on the
// tensor cores through mma.sync (f32 accumulation): bf16 inputs for groups of up to 64
// query rows per kv head (above 16: the wide kernel), FP8 E4M3 caches (widened to f16)
// and f32 inputs (three TF32 products per f32 product) for groups of up to 16 and 8 rows.
//
// Why tensor cores here: with G query heads sharing one KV head, every KV element
// feeds G multiply-adds for the scores and G for the output, i.e. G FLOP per KV byte.
// At G = 8 and ~7 TB/s that is ~55 TFLOP/s of FMA work, about 75% of the CUDA-core
// FP32 rate of a GB300, so the CUDA-core kernel (fd_partial_simt.cuh) is co-limited
// by arithmetic.  The same work is under 20% of the legacy tensor-core (mma.sync)
// rate, which leaves the pass bound by HBM, as it should be.
//
// Memory side: the TMA producer warp and stage ring of fd_pipeline.cuh (128-byte
// swizzled K/V tiles).  Compute side, per consumer warp and per 16-token chunk:
//   S^T[16 tok, 8 rows] = K_chunk[16, d] . Q^T[d, 8]           (tokens in M, query rows in
//                                                                N: G = 8 fills N exactly;
//                                                                multi-token decode adds
//                                                                Q x G rows, up to 16)
//   scores -> base-2 logits, mask (-inf), online-softmax max / rescale
//   P^T = movmatrix.trans(bf16(2^(S - m)))                      (register transpose)
//   O^T[d, 8] += V_chunk^T[d, 16 tok] . P^T[16 tok, 8 heads]    (V^T via ldmatrix.trans)
// which is the FlashAttention update of "AI Infra: math and infra optimisation in large
// models", section 2.6 (S = Q K^T per KV block; rescale the running sum and output by
// exp(m_old - m_new); add exp(S - m_new) V), run inside one KV split of
// Flash-Decoding (same section, "Flash-Decoding Split-K").
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fd_epilogue.cuh"

namespace fd {

namespace {

// G: query rows a consumer warp works on (the whole group, padded to a power of two;
// with WIDE, the warp's quarter of a group of 32 or 64 rows).  WIDE: each consumer warp
// takes all tokens of every tile for its own rows, instead of a quarter of the tokens
// for all rows.
// F32: q, K and V stored as f32, multiplied on the tensor cores as three TF32 products
// (see split_tf32), for groups of up to 8 rows.
// Tiles of its split a CTA prefetches into L2 before it may read its inputs
// (prefetch_first_tiles), and how many tiles before the end of its loop the consumers
// let the next kernel of the stream launch.  Measured on the 128K GQA workload (graphs
// of back-to-back steps): no prefetch 78.5 us, 4 tiles 75.5 us, 8 tiles 75.0 us,
// 12 tiles 76.1 us; the early trigger helps the short MHA step (40.1 -> 38.8 us).
constexpr int kPrefetchTiles = 8;
// Head-group tiles (16 tokens x 4 kv heads, 32 KB), paged: ragged paged workload (16-token
// pages) 135.6 us without, 134.7 us with 8, 133.6 us with 4.
constexpr int kPrefetchHeadTiles = 4;
constexpr int kTriggerTiles = 4;

template <int D_, int G_, bool KV8_ = false, bool PERSIST_ = false, bool WIDE_ = false,
          bool F32_ = false>
struct MmaShape {
  static constexpr int D = D_;
  static constexpr int G = G_;
  static constexpr bool KV8 = KV8_;                        // K/V stored as FP8 E4M3 codes
  static constexpr bool WIDE = WIDE_;
  static constexpr bool F32 = F32_;
  static_assert(!(WIDE && KV8 && G_ > 8), "wide groups: FP8 up to 8 rows a warp");
  static_assert(!(F32 && (KV8 || PERSIST_ || WIDE_ || G_ > 8)),
                "f32 inputs: grid schedule, up to 8 rows");
  static constexpr int NT = G > 8 ? 2 : 1;                 // n-tiles of 8 heads
  static constexpr int ROW_BYTES = D * (F32 ? 4 : (KV8 ? 1 : 2));
  static constexpr int TT = kTileBytes / ROW_BYTES;        // 64 (bf16 d=128), 128 (d=64 or
                                                           // fp8), 32 (f32 d=128)
  static constexpr int LINES = ROW_BYTES / 128;
  static constexpr int NCW = F32 ? TT / 16 : 4;            // consumer warps (f32 d=128: 2)
  static constexpr int ROWS_PER_WARP = WIDE ? TT : TT / NCW;   // token rows of a warp per tile
  static constexpr int CHUNKS = ROWS_PER_WARP / 16;        // 16-token chunks per warp per tile
  // chunks sharing one softmax update (wide groups of 8 rows a warp: the whole tile)
  static constexpr int JOINT = (WIDE && NT == 1) ? CHUNKS : (CHUNKS < 2 ? CHUNKS : 2);
  static constexpr int KSTEPS = F32 ? D / 8 : D / 16;     // k-steps of the QK^T product
  static constexpr int QLO = F32 ? KSTEPS : 1;             // TF32 residual fragments of q
  static constexpr int MTILES = D / 16;                    // m-tiles of the PV product
  // Persistent schedule: the same two CTAs per SM, each taking items from a queue; an
  // item's epilogue uses the ring stage of its last tile as merge scratch (the other
  // stages, and the other CTA of the SM, keep streaming meanwhile).
  static constexpr bool PERSIST = PERSIST_;
  static constexpr int STAGES = 3;
  static constexpr int THREADS = (NCW + 1) * 32;
  static constexpr int MERGE_BYTES = NCW * G * D * 4 + 2 * NCW * G * 4;
  static_assert(MERGE_BYTES <= STAGES * 2 * kTileBytes, "merge scratch fits the stages");
  static_assert(NCW * G * D * 4 <= 2 * kTileBytes && NCW * G <= 64,
                "persistent merge scratch fits one stage and the control block");
  static constexpr size_t RING_BYTES = (size_t)STAGES * 2 * kTileBytes;
  static constexpr size_t SMEM_BYTES =
      1024 + RING_BYTES + (PERSIST ? sizeof(PersistCtl<STAGES>) : sizeof(PipeCtl<STAGES>));
  static_assert(2 * (SMEM_BYTES + 1024) <= 228 * 1024, "two CTAs per SM");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D = A . B + D, m16n8k16, bf16 inputs, f32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A . B + D, m16n8k8, TF32 inputs, f32 accumulators (the f32 path).
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// An f32 value as a TF32 pair hi + lo.  hi: x rounded to the nearest TF32 value (10
// mantissa bits, ties away from zero), by adding half a TF32 unit to the bit pattern and
// clearing the 13 low bits (a carry into the exponent is the correct rounding up to the
// next binade).  lo = x - hi, exact in f32 and at most half a TF32 unit of x (2^-11 |x|);
// the mma reads it as TF32 (its low 13 bits do not take part), an error below 2^-21 |x|.  With a = ah + al and b = bh + bl, ah bh + ah bl + al bh then carries about
// 21 bits of each product (al bl, ~2^-22 relative, is dropped): f32 accuracy for this
// pass from three TF32 tensor-core products, at three integer/float ops per split.
// Non-finite inputs only occur in masked slots, whose scores are replaced by -inf and
// whose V rows are zeroed before use.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = (__float_as_uint(x) + 0x1000u) & 0xffffe000u;
  lo = __float_as_uint(x - __uint_as_float(hi));
}

// D = A . B + D, m16n8k16, f16 inputs, f32 accumulators (the FP8 KV path).
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two FP8 E4M3 codes (low byte -> low half) to an f16x2; exact (every E4M3 value is an
// f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes_in_low_16) {
  uint32_t y;
  const uint16_t x = (uint16_t)(two_codes_in_low_16 & 0xffffu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(y) : "h"(x));
  return y;
}

// Byte permute: bytes of {b:a} picked by the selector nibbles (prmt.b32).
__device__ __forceinline__ uint32_t byte_perm(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Pack two f32 into a bf16x2 (round to nearest even); `lo` goes to the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Per-consumer-warp state and tile math of the tensor-core partial pass: the query
// fragments of one (b, kv head) group, the online-softmax state (m, l) and the O^T
// accumulator of this warp's share of the tokens.  Used per split by the grid and
// head-group kernels and per work item by the persistent kernel.
template <class SH>
struct Consumer {
  static constexpr int NT = SH::NT;
  uint32_t qb[NT][SH::KSTEPS][2];  // Q^T B-fragments (f32 path: the TF32 high parts)
  uint32_t qlo[NT][SH::QLO][2];    // f32 path: the TF32 residuals
  int64_t lim[NT][2];              // causal key bound of this thread's two columns per n-tile
  float m[NT][2], l[NT][2];        // per column (query row nt * 8 + qc + {0, 1})
  float acc[NT][SH::MTILES][4];    // O^T fragments
  float sl2, vsc;
  int64_t kmin;                    // smallest causal key bound of the warp's rows
  int row0;                        // first query row of the group this warp works on

  // Load the group's query fragments and reset the state.
  //   B fragments of Q^T (k = dim, n = row), bf16 as stored: b0 holds dims 16 kk + qc,
  //   +1 of row nt * 8 + qr; b1 the same 8 dims further.  Rows >= n_rows are 0.
  //   FP8 KV: the k index of the QK^T mma is a permutation of the dims (see tile()): in
  //   a 16-dim step, fragment columns (2c, 2c+1) hold dims (4c, 4c+1) and columns
  //   (2c+8, 2c+9) hold dims (4c+2, 4c+3), c = lane % 4.  q is converted to f16 (exact
  //   for bf16 values in f16's range) with the same permutation.
  //   F32: m16n8k8 B fragments, b0 = dim 8 kk + c, b1 = dim 8 kk + c + 4 of row qr, each
  //   split into TF32 high part (qb) and residual (qlo).
  __device__ __forceinline__ void start(const Params& p, int b, int g, int64_t L, int lane,
                                        int first_row = 0) {
    const int qr = lane >> 2, qc = (lane & 3) * 2;
    row0 = first_row;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = row0 + nt * 8 + qr;
      const bool live = h < p.n_rows;
      if constexpr (SH::F32) {
        const float* qf = reinterpret_cast<const float*>(p.q) + q_offset(p, b, g, live ? h : 0);
        const int c = lane & 3;
#pragma unroll
        for (int kk = 0; kk < SH::KSTEPS; ++kk) {
          split_tf32(live ? qf[kk * 8 + c] : 0.f, qb[nt][kk][0], qlo[nt][kk][0]);
          split_tf32(live ? qf[kk * 8 + c + 4] : 0.f, qb[nt][kk][1], qlo[nt][kk][1]);
        }
      } else {
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          reinterpret_cast<const __nv_bfloat16*>(p.q) +
          q_offset(p, b, g, live ? h : 0));           // never address past the group
#pragma unroll
      for (int kk = 0; kk < SH::KSTEPS; ++kk) {
        uint32_t lo, hi;
        if constexpr (SH::KV8) {
          const uint32_t w0 = qrow[(kk * 16 + 2 * qc) / 2], w1 = qrow[(kk * 16 + 2 * qc + 2) / 2];
          lo = pack_f16x2(bf16lo_to_f32(w0), bf16hi_to_f32(w0));
          hi = pack_f16x2(bf16lo_to_f32(w1), bf16hi_to_f32(w1));
        } else {
          lo = qrow[(kk * 16 + qc) / 2];
          hi = qrow[(kk * 16 + qc + 8) / 2];
        }
        qb[nt][kk][0] = live ? lo : 0u;
        qb[nt][kk][1] = live ? hi : 0u;
      }
      }
      lim[nt][0] = key_bound(p, L, row0 + nt * 8 + qc);
      lim[nt][1] = key_bound(p, L, row0 + nt * 8 + qc + 1);
      m[nt][0] = m[nt][1] = kNegInf;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < SH::MTILES; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][mt][e] = 0.f;
    }
    kmin = key_bound(p, L, row0);
    // FP8 KV: per-kv-head dequantisation scales fold into the score scale and output.
    const float ksc = (SH::KV8 && p.k_scale != nullptr) ? p.k_scale[g] : 1.f;
    vsc = (SH::KV8 && p.v_scale != nullptr) ? p.v_scale[g] : 1.f;
    sl2 = p.scale_log2 * ksc;
  }

  // One K/V tile in shared memory: this warp's ROWS_PER_WARP token rows of it (all of
  // them with WIDE).  Valid tokens are [lo, hi) minus invalid pages (`bad`); each query
  // row also keeps only keys below its causal bound.
  __device__ __forceinline__ void tile(const Params& p, uint8_t* kt, uint8_t* vt, int64_t t0,
                                       int64_t lo, int64_t hi, uint32_t bad, int warp, int lane,
                                       uint32_t lb, bool multi_page) {
    const int qr = lane >> 2;
    const int lm = lane >> 3, lr = lane & 7;          // ldmatrix: matrix i / 8, row i % 8
    const int r0 = SH::WIDE ? 0 : warp * SH::ROWS_PER_WARP;   // warp's first row in the tile

    // Rows outside [lo, hi) or on an invalid page: their V rows may be stale (NaN) and
    // 0 * NaN is NaN inside the MMA, so they must read as 0.  Only boundary tiles.  A
    // warp that owns its rows zeroes them in shared memory; with WIDE every warp reads
    // every row, so the V fragments are masked in registers instead (below).
    const bool clean = t0 + r0 >= lo && t0 + r0 + SH::ROWS_PER_WARP <= hi && bad == 0;
    if (!SH::WIDE && !clean) {
      for (int r = 0; r < SH::ROWS_PER_WARP; ++r) {
        const int row = r0 + r;
        const int64_t tok = t0 + row;
        const int pslot = multi_page ? (row >> p.log2_page) : 0;
        const bool valid = tok >= lo && tok < hi && !((bad >> pslot) & 1u);
        if (!valid) {
          for (int c = lane; c < SH::ROW_BYTES / 16; c += 32)
            *reinterpret_cast<uint4*>(vt + tile_chunk<SH::LINES>(row, c, lb)) = make_uint4(0, 0, 0, 0);
        }
      }
      // These generic-proxy stores must be ordered before the next TMA write of the stage.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }

    // JOINT 16-token chunks at a time go through the online softmax together: all their
    // QK^T products first (independent mma chains), one max and one rescale, then all
    // their PV products.
    // A row needs masking only on a boundary tile (split range, invalid page) or where
    // a query's causal bound falls inside the warp's rows; kmin is the smallest bound.
    const bool full = clean && t0 + r0 + SH::ROWS_PER_WARP <= kmin;
#pragma unroll
    for (int cg = 0; cg < SH::CHUNKS; cg += SH::JOINT) {
    float s[SH::JOINT][NT][4];
#pragma unroll
    for (int ch = 0; ch < SH::JOINT; ++ch) {
      const int rb = r0 + (cg + ch) * 16;             // first row of this 16-token chunk
      // ---- S^T = K . Q^T  (A = K rows rb..rb+15 via ldmatrix, swizzled tile)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) s[ch][nt][0] = s[ch][nt][1] = s[ch][nt][2] = s[ch][nt][3] = 0.f;
      const int arow = rb + lr + (lm & 1) * 8;
      if constexpr (SH::KV8) {
        // A 16-byte chunk holds 16 dims: one ldmatrix.x4 (chunks c, c + 1, rows 0-7 and
        // 8-15) feeds two k-steps.  A register holds dims 4c'..4c'+3 of one row; its low
        // half gives fragment columns (2c', 2c'+1), its high half (2c'+8, 2c'+9).
#pragma unroll
        for (int kk = 0; kk < SH::KSTEPS; kk += 2) {
          const int c16 = kk + (lm >> 1);
          uint32_t r[4];
          ldsm_x4(smem_addr(kt) + tile_chunk<SH::LINES>(arow, c16, lb), r);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t rr0 = r[2 * u], rr1 = r[2 * u + 1];
            const uint32_t a[4] = {e4m3x2_to_f16x2(rr0), e4m3x2_to_f16x2(rr1),
                                   e4m3x2_to_f16x2(rr0 >> 16), e4m3x2_to_f16x2(rr1 >> 16)};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_f16(s[ch][nt], a, qb[nt][kk + u][0], qb[nt][kk + u][1]);
          }
        }
      } else if constexpr (SH::F32) {
        // A 16-byte chunk holds 4 dims: ldmatrix.x4 over chunks 2 kk, 2 kk + 1 and rows
        // 0-7, 8-15 gives exactly the m16n8k8 A fragment (a register is one f32 of row
        // qr or qr + 8 at dim 8 kk + c or + 4).  K . Q^T = Kh Qh + Kh Ql + Kl Qh.  Each
        // product and each parity of kk has its own accumulator (six independent mma
        // chains of KSTEPS / 2), summed at the end.
        float sp[3][2][NT][4];
#pragma unroll
        for (int j = 0; j < 3; ++j)
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) sp[j][u][nt][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < SH::KSTEPS; ++kk) {
          const int c16 = kk * 2 + (lm >> 1);
          uint32_t r[4], ah[4], al[4];
          ldsm_x4(smem_addr(kt) + tile_chunk<SH::LINES>(arow, c16, lb), r);
#pragma unroll
          for (int i = 0; i < 4; ++i) split_tf32(__uint_as_float(r[i]), ah[i], al[i]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_tf32(sp[0][kk & 1][nt], ah, qlo[nt][kk][0], qlo[nt][kk][1]);
            mma_tf32(sp[1][kk & 1][nt], al, qb[nt][kk][0], qb[nt][kk][1]);
            mma_tf32(sp[2][kk & 1][nt], ah, qb[nt][kk][0], qb[nt][kk][1]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            s[ch][nt][e] = ((sp[0][0][nt][e] + sp[0][1][nt][e]) +
                            (sp[1][0][nt][e] + sp[1][1][nt][e])) +
                           (sp[2][0][nt][e] + sp[2][1][nt][e]);
      } else {
#pragma unroll
        for (int kk = 0; kk < SH::KSTEPS; ++kk) {
          const int c16 = kk * 2 + (lm >> 1);         // 16-byte chunk of the row
          uint32_t a[4];
          ldsm_x4(smem_addr(kt) + tile_chunk<SH::LINES>(arow, c16, lb), a);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_bf16(s[ch][nt], a, qb[nt][kk][0], qb[nt][kk][1]);
        }
      }
    }

    // ---- mask and scale: element e of s[ch][nt] is (token rb + qr + 8 (e >> 1),
    //      row nt * 8 + qc + (e & 1)); excluded tokens get -inf.
    if (full) {
#pragma unroll
      for (int ch = 0; ch < SH::JOINT; ++ch)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[ch][nt][e] *= sl2;
    } else {
#pragma unroll
      for (int ch = 0; ch < SH::JOINT; ++ch) {
        const int rb = r0 + (cg + ch) * 16;
        bool vrow[2];
        int64_t vtok[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int row = rb + qr + 8 * hh;
          const int64_t tok = t0 + row;
          const int pslot = multi_page ? (row >> p.log2_page) : 0;
          vrow[hh] = tok >= lo && tok < hi && !((bad >> pslot) & 1u);
          vtok[hh] = tok;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            s[ch][nt][e] = (vrow[e >> 1] && vtok[e >> 1] < lim[nt][e & 1]) ? s[ch][nt][e] * sl2
                                                                             : kNegInf;
      }
    }

    uint32_t pb[SH::JOINT][NT][2];                    // P^T fragments (b0/b1 of the PV mma)
    // F32: m16n8k8 P^T fragments per 8-token half kk of the chunk, TF32 high parts and
    // residuals.  The PV k index t <-> token 2t, t + 4 <-> token 2t + 1 of the half.
    uint32_t pf[SH::F32 ? SH::JOINT : 1][NT][2][2], pfl[SH::F32 ? SH::JOINT : 1][NT][2][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      // max per column over the chunks' rows: in-thread, then lanes of equal qc
      float mx0 = kNegInf, mx1 = kNegInf;
#pragma unroll
      for (int ch = 0; ch < SH::JOINT; ++ch) {
        mx0 = fmaxf(mx0, fmaxf(s[ch][nt][0], s[ch][nt][2]));
        mx1 = fmaxf(mx1, fmaxf(s[ch][nt][1], s[ch][nt][3]));
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
      if (mn0 > m[nt][0] || mn1 > m[nt][1]) {         // rescale the running state
        const float c0 = (mn0 == kNegInf) ? 1.f : ex2(m[nt][0] - mn0);
        const float c1 = (mn1 == kNegInf) ? 1.f : ex2(m[nt][1] - mn1);
        l[nt][0] *= c0;
        l[nt][1] *= c1;
#pragma unroll
        for (int mt = 0; mt < SH::MTILES; ++mt) {
          acc[nt][mt][0] *= c0;
          acc[nt][mt][1] *= c1;
          acc[nt][mt][2] *= c0;
          acc[nt][mt][3] *= c1;
        }
        m[nt][0] = mn0;
        m[nt][1] = mn1;
      }
#pragma unroll
      for (int ch = 0; ch < SH::JOINT; ++ch) {
        float pr[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x = s[ch][nt][e];
          pr[e] = (x == kNegInf) ? 0.f : ex2(x - m[nt][e & 1]);
        }
        l[nt][0] += pr[0] + pr[2];
        l[nt][1] += pr[1] + pr[3];
        // P rows (tokens qr, qr + 8) x columns (qc, qc + 1) -> transpose to P^T fragments.
        if constexpr (SH::F32) {
          // b0 of lane (g, c) is P[token 8 kk + 2c][row g], held by lane 8c + g / 2 as its
          // element 2 kk + (g & 1); b1 is token 2c + 1, held by lane 8c + 4 + g / 2.
          const int src0 = 8 * (lane & 3) + (qr >> 1);
          const bool odd = qr & 1;
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const float x0 = __shfl_sync(0xffffffffu, pr[2 * kk], src0 + 4 * j);
              const float x1 = __shfl_sync(0xffffffffu, pr[2 * kk + 1], src0 + 4 * j);
              split_tf32(odd ? x1 : x0, pf[ch][nt][kk][j], pfl[ch][nt][kk][j]);
            }
          }
        } else if constexpr (SH::KV8) {                      // f16 P for the f16 PV mma
          pb[ch][nt][0] = movmatrix_trans(pack_f16x2(pr[0], pr[1]));
          pb[ch][nt][1] = movmatrix_trans(pack_f16x2(pr[2], pr[3]));
        } else {
          pb[ch][nt][0] = movmatrix_trans(pack_bf16x2(pr[0], pr[1]));
          pb[ch][nt][1] = movmatrix_trans(pack_bf16x2(pr[2], pr[3]));
        }
      }
    }

    // ---- O^T += V^T . P^T
#pragma unroll
    for (int ch = 0; ch < SH::JOINT; ++ch) {
      const int rb = r0 + (cg + ch) * 16;
      if constexpr (SH::F32) {
        // m16n8k8 A fragment of V^T from two 8-byte loads: m-row qr <-> dim 16 mt + 2 qr,
        // m-row qr + 8 <-> dim 16 mt + 2 qr + 1 (undone when the output is written), k
        // index c <-> token 2c and c + 4 <-> token 2c + 1.  A half-warp's 16 loads cover
        // 16 distinct 8-byte slots of the swizzled rows: no bank conflicts.
        const int c = lane & 3;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int row = rb + 8 * kk + 2 * c;
#pragma unroll
          for (int mt = 0; mt < SH::MTILES; ++mt) {
            const int dim = mt * 16 + 2 * qr;
            const uint32_t off = (uint32_t)(dim & 3) * 4u;
            const uint2 x = *reinterpret_cast<const uint2*>(
                vt + tile_chunk<SH::LINES>(row, dim >> 2, lb) + off);
            const uint2 y = *reinterpret_cast<const uint2*>(
                vt + tile_chunk<SH::LINES>(row + 1, dim >> 2, lb) + off);
            const uint32_t a[4] = {x.x, x.y, y.x, y.y};
            uint32_t ah[4], al[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) split_tf32(__uint_as_float(a[i]), ah[i], al[i]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_tf32(acc[nt][mt], ah, pfl[ch][nt][kk][0], pfl[ch][nt][kk][1]);
              mma_tf32(acc[nt][mt], al, pf[ch][nt][kk][0], pf[ch][nt][kk][1]);
              mma_tf32(acc[nt][mt], ah, pf[ch][nt][kk][0], pf[ch][nt][kk][1]);
            }
          }
        }
      } else if constexpr (SH::KV8) {
        // ldmatrix.trans over 16-bit pairs of codes: matrix j covers tokens
        // rb + 8 (j & 1) .. +7 of chunk (m-tile) mt + (j >> 1); a register holds tokens
        // (qc, qc+1) x dims (2 qr, 2 qr + 1).  Regrouped by dim (prmt) and widened, it
        // gives the A fragment of V^T with m-row qr <-> dim 2 qr and m-row qr + 8 <->
        // dim 2 qr + 1 of the 16-dim tile (undone when the output is written).
        const int vtok_addr = rb + lr + (lm & 1) * 8;
        // WIDE: every warp reads every row, so V rows outside [lo, hi) or on an invalid
        // page are masked in registers (after widening: their codes may be NaN).  a[0],
        // a[1] hold tokens 2c, 2c + 1 of the chunk (low, high half), a[2], a[3] tokens
        // 2c + 8, 2c + 9, c = lane % 4 -- as in the bf16 branch below.
        uint32_t vmask[2] = {0xffffffffu, 0xffffffffu};
        if (SH::WIDE && !clean) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t mk = 0u;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int row = rb + 8 * hh + 2 * (lane & 3) + u;
              const int64_t tok = t0 + row;
              const int pslot = multi_page ? (row >> p.log2_page) : 0;
              if (tok >= lo && tok < hi && !((bad >> pslot) & 1u)) mk |= 0xffffu << (16 * u);
            }
            vmask[hh] = mk;
          }
        }
#pragma unroll
        for (int mt = 0; mt < SH::MTILES; mt += 2) {
          const int c16 = mt + (lm >> 1);
          uint32_t r[4];
          ldsm_x4_trans(smem_addr(vt) + tile_chunk<SH::LINES>(vtok_addr, c16, lb), r);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t x0 = byte_perm(r[2 * u], 0u, 0x3120u);       // tokens 0-7
            const uint32_t x1 = byte_perm(r[2 * u + 1], 0u, 0x3120u);   // tokens 8-15
            uint32_t a[4] = {e4m3x2_to_f16x2(x0), e4m3x2_to_f16x2(x0 >> 16),
                             e4m3x2_to_f16x2(x1), e4m3x2_to_f16x2(x1 >> 16)};
            if (SH::WIDE && !clean) {
              a[0] &= vmask[0];
              a[1] &= vmask[0];
              a[2] &= vmask[1];
              a[3] &= vmask[1];
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_f16(acc[nt][mt + u], a, pb[ch][nt][0], pb[ch][nt][1]);
          }
        }
      } else {
        // A = V^T via ldmatrix.trans: matrix j covers tokens rb + 8 (j >> 1) .. +7 and
        // dims 16 mt + 8 (j & 1) .. +7; a register holds tokens rb + 8 (j >> 1) + 2 c and
        // + 1 (low, high half), c = lane % 4, at one dim.
        const int vrow_addr = rb + lr + (lm >> 1) * 8;
        uint32_t vmask[2] = {0xffffffffu, 0xffffffffu};   // tokens +0/+1 and +8/+9
        if (SH::WIDE && !clean) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t mk = 0u;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int row = rb + 8 * hh + 2 * (lane & 3) + u;
              const int64_t tok = t0 + row;
              const int pslot = multi_page ? (row >> p.log2_page) : 0;
              if (tok >= lo && tok < hi && !((bad >> pslot) & 1u)) mk |= 0xffffu << (16 * u);
            }
            vmask[hh] = mk;
          }
        }
#pragma unroll
        for (int mt = 0; mt < SH::MTILES; ++mt) {
          const int c16 = mt * 2 + (lm & 1);
          uint32_t a[4];
          ldsm_x4_trans(smem_addr(vt) + tile_chunk<SH::LINES>(vrow_addr, c16, lb), a);
          if (SH::WIDE && !clean) {
            a[0] &= vmask[0];
            a[1] &= vmask[0];
            a[2] &= vmask[1];
            a[3] &= vmask[1];
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_bf16(acc[nt][mt], a, pb[ch][nt][0], pb[ch][nt][1]);
        }
      }
    }
    }                                                  // chunk groups
  }

  // End of a split: sum l over the 8 lanes that share a column (they saw different
  // tokens) and write this warp's (m, l, acc) into the merge scratch
  // macc [NCW][G][D] (macc_index), mm [NCW][G], ml [NCW][G].
  __device__ __forceinline__ void store(const Params& p, float* macc, float* mm, float* ml,
                                        int warp, int lane) {
    constexpr int G = SH::G;
    const int qr = lane >> 2, qc = (lane & 3) * 2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], off);
        l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], off);
      }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = nt * 8 + qc + e;
        if (h < p.n_rows) {
#pragma unroll
          for (int mt = 0; mt < SH::MTILES; ++mt) {
            // m-rows qr, qr + 8 of tile mt are dims 16 mt + (qr, qr + 8), or with FP8 KV
            // or f32 dims 16 mt + (2 qr, 2 qr + 1); the V scale applies to the whole output.
            constexpr bool PAIRED = SH::KV8 || SH::F32;
            const int d0 = PAIRED ? 2 * qr : qr, d1 = PAIRED ? 2 * qr + 1 : qr + 8;
            macc[macc_index<G, SH::D>(warp, h, mt * 16 + d0)] = acc[nt][mt][e] * vsc;
            macc[macc_index<G, SH::D>(warp, h, mt * 16 + d1)] = acc[nt][mt][2 + e] * vsc;
          }
          if (qr == 0) {
            mm[warp * G + h] = m[nt][e];
            ml[warp * G + h] = l[nt][e];
          }
        }
      }
    }
  }

  // Whether store_own can write a single split's result as the output (Params::direct):
  // not for 16 rows per warp, where the head-group and wide kernels sit at their
  // register cap (the direct branch made them spill); mma_writes_direct tells the host.
  __host__ __device__ static constexpr bool direct_ok() { return SH::G <= 8; }

  // End of a split when this warp alone saw all of it (head-group tiles: one warp per kv
  // head): write O_i = acc / l and LSE_i = (m + log2 l) ln 2 of the warp's rows directly,
  // the single-warp case of merge_warps_and_store.
  __device__ __forceinline__ void store_own(const Params& p, int b, int g, int split, int lane) {
    const int qr = lane >> 2, qc = (lane & 3) * 2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], off);
        l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], off);
      }
    constexpr bool PAIRED = SH::KV8 || SH::F32;
    const int d0 = PAIRED ? 2 * qr : qr, d1 = PAIRED ? 2 * qr + 1 : qr + 8;
    if constexpr (direct_ok()) {
      if (p.direct) {               // the row of out; a row without keys gets zeros
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = row0 + nt * 8 + qc + e;
            if (h >= p.n_rows) continue;
            const float L = l[nt][e];
            const int64_t o = out_elem(p, b, g, h);
#pragma unroll
            for (int mt = 0; mt < SH::MTILES; ++mt) {
              put_out(p, o + mt * 16 + d0, L > 0.f ? acc[nt][mt][e] * vsc / L : 0.f);
              put_out(p, o + mt * 16 + d1, L > 0.f ? acc[nt][mt][2 + e] * vsc / L : 0.f);
            }
            if (qr == 0)
              put_lse(p, b, g, h, split,
                      L > 0.f ? (m[nt][e] + lg2_approx(L)) * 0.6931471805599453f : kNegInf);
          }
        }
        return;
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = row0 + nt * 8 + qc + e;
        if (h >= p.n_rows) continue;
        const int64_t row = flat_row(p, b, g, h);
        const float L = l[nt][e];
        if (L > 0.f) {
          float* o = p.o_part + (row * p.S + split) * SH::D;
#pragma unroll
          for (int mt = 0; mt < SH::MTILES; ++mt) {
            o[mt * 16 + d0] = acc[nt][mt][e] * vsc / L;
            o[mt * 16 + d1] = acc[nt][mt][2 + e] * vsc / L;
          }
          if (qr == 0) p.lse_part[row * p.S + split] = (m[nt][e] + lg2_approx(L)) * 0.6931471805599453f;
        } else if (qr == 0) {
          p.lse_part[row * p.S + split] = kNegInf;
        }
      }
    }
  }
};

// ---------------------------------------------------------------- grid schedule
// One CTA per (split, kv head, row); two CTAs per SM.
template <class SH>
__global__ void __launch_bounds__(SH::THREADS, 2)
    fd_partial_mma_kernel(const __grid_constant__ CUtensorMap tk,
                          const __grid_constant__ CUtensorMap tv,
                          const __grid_constant__ Params p) {
  constexpr int G = SH::G, TT = SH::TT, STAGES = SH::STAGES;
  if (threadIdx.x == SH::NCW * 32) {
    // Paged caches with pages of at least a tile: page ids from the block table (not
    // with 16 query rows per kv head, where the extra registers would spill).  128K GQA
    // in 64-token pages: 80.4 -> 77.9 us per step.
    if constexpr (SH::G <= 8) {
      if (p.block_table != nullptr && p.page_size >= TT)
        prefetch_first_pages<TT>(p, &tk, &tv, kPrefetchTiles, (int)blockIdx.y);
    }
    prefetch_first_tiles<TT>(p, &tk, &tv, kPrefetchTiles, (int)blockIdx.y);
  }
  pdl_wait();                       // inputs of this step are visible
  const SplitInfo si = split_info<TT>(p);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  auto* ctl = reinterpret_cast<PipeCtl<STAGES>*>(stages + SH::RING_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (si.n_tiles == 0) {            // empty split: weight 0 in the merge, nothing to load
    write_empty_split(p, si, threadIdx.x);
    pdl_trigger();
    if (p.counters != nullptr && warp < SH::NCW)
      arrive_and_merge<SH::D, SH::NCW>(p, si, threadIdx.x, &ctl->last);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_addr(&ctl->full[s]), 1);
      mbar_init(smem_addr(&ctl->empty[s]), SH::NCW);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == SH::NCW) {            // ---------------- producer warp
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
    produce_tiles<TT, STAGES>(p, si, &tk, &tv, stages, ctl, lane);
    pdl_trigger();
    return;
  }

  // ---------------------------------------------------- consumer warps
  Consumer<SH> c;
  c.start(p, si.b, si.g, si.L, lane);
  const bool multi_page = p.page_size > 0 && p.page_size < TT;
  const uint32_t lb = (uint32_t)p.log2_box;
  bool aborted = false;
  // The next kernel of the stream may launch once kTriggerTiles tiles are left: its CTAs
  // take free slots and prefetch their first tiles while this split finishes.
  const int trigger_at = si.n_tiles > kTriggerTiles ? si.n_tiles - kTriggerTiles : 0;
  int n = 0;
  for (; n < si.n_tiles; ++n) {
    if (n == trigger_at) pdl_trigger();
    const int stage = n % STAGES;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_addr(&ctl->full[stage]), (n / STAGES) & 1);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        ctl->abort = 1;
        atomicOr(p.flags, kDevFlagTimeout);
      }
      aborted = true;
      break;
    }
    uint8_t* kt = stages + (size_t)stage * 2 * kTileBytes;
    c.tile(p, kt, kt + kTileBytes, si.T0 + (int64_t)n * TT, si.lo, si.hi, ctl->bad[stage], warp,
           lane, lb, multi_page);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl->empty[stage]));
  }
  if (n < trigger_at) pdl_trigger();    // the loop ended before the trigger (an abort)

  named_bar_sync(1, SH::NCW * 32);
  if (aborted || *reinterpret_cast<volatile int32_t*>(&ctl->abort)) {
    if (warp == 0) write_empty_split(p, si, threadIdx.x);
    if (p.counters != nullptr) arrive_and_merge<SH::D, SH::NCW>(p, si, threadIdx.x, &ctl->last);
    return;
  }
  float* macc = reinterpret_cast<float*>(stages);                 // [NCW][G][D], ring drained
  float* mm = macc + SH::NCW * G * SH::D;                         // [NCW][G]
  float* ml = mm + SH::NCW * G;                                   // [NCW][G]
  c.store(p, macc, mm, ml, warp, lane);
  named_bar_sync(1, SH::NCW * 32);
  merge_warps_and_store<G, SH::D, SH::NCW>(p, si, macc, mm, ml, threadIdx.x, [] {
    named_bar_sync(1, SH::NCW * 32);
    return true;
  });
  if (p.counters != nullptr) arrive_and_merge<SH::D, SH::NCW>(p, si, threadIdx.x, &ctl->last);
}

// ---------------------------------------------------------------- wide groups
// Query groups of 17 to 64 rows (Q query tokens x G heads of a kv head, or G > 16):
// one CTA per (split, kv head, row) as in the grid schedule, but consumer warp w works
// on rows w G .. w G + G - 1 (G = 8 or 16 here) over every token of each tile, so a
// warp's state covers its rows for the whole split and it writes their partials itself
// (no cross-warp merge).  Each K/V tile is read from shared memory by all four warps.
// Two CTAs of 160 threads per SM leave 204 registers per thread; __launch_bounds__
// would budget for 192-thread CTAs and cap at 168, which spills the wide accumulators.
template <class SH>
__global__ void __maxnreg__(200)
    fd_partial_wide_kernel(const __grid_constant__ CUtensorMap tk,
                           const __grid_constant__ CUtensorMap tv,
                           const __grid_constant__ Params p) {
  constexpr int TT = SH::TT, STAGES = SH::STAGES;
  static_assert(SH::WIDE, "wide shape");
  if (threadIdx.x == SH::NCW * 32) prefetch_first_tiles<TT>(p, &tk, &tv, kPrefetchTiles, (int)blockIdx.y);
  pdl_wait();                       // inputs of this step are visible
  const SplitInfo si = split_info<TT>(p);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  auto* ctl = reinterpret_cast<PipeCtl<STAGES>*>(stages + SH::RING_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (si.n_tiles == 0) {            // empty split: weight 0 in the merge, nothing to load
    write_empty_split(p, si, threadIdx.x);
    pdl_trigger();
    if (p.counters != nullptr && warp < SH::NCW)
      arrive_and_merge<SH::D, SH::NCW>(p, si, threadIdx.x, &ctl->last);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_addr(&ctl->full[s]), 1);
      mbar_init(smem_addr(&ctl->empty[s]), SH::NCW);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == SH::NCW) {            // ---------------- producer warp
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
    produce_tiles<TT, STAGES>(p, si, &tk, &tv, stages, ctl, lane);
    pdl_trigger();
    return;
  }

  Consumer<SH> c;
  c.start(p, si.b, si.g, si.L, lane, warp * SH::G);
  const bool multi_page = p.page_size > 0 && p.page_size < TT;
  const uint32_t lb = (uint32_t)p.log2_box;
  bool aborted = false;
  for (int n = 0; n < si.n_tiles; ++n) {
    const int stage = n % STAGES;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_addr(&ctl->full[stage]), (n / STAGES) & 1);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        ctl->abort = 1;
        atomicOr(p.flags, kDevFlagTimeout);
      }
      aborted = true;
      break;
    }
    uint8_t* kt = stages + (size_t)stage * 2 * kTileBytes;
    c.tile(p, kt, kt + kTileBytes, si.T0 + (int64_t)n * TT, si.lo, si.hi, ctl->bad[stage], warp,
           lane, lb, multi_page);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl->empty[stage]));
  }
  pdl_trigger();
  if (aborted) {                    // this warp's rows of the split: weight 0
    const int h = warp * SH::G + lane;
    if (lane < SH::G && h < p.n_rows) put_empty_row<Consumer<SH>::direct_ok()>(p, si.b, si.g, h, si.split);
  } else {
    c.store_own(p, si.b, si.g, si.split, lane);
  }
  if (p.counters != nullptr) arrive_and_merge<SH::D, SH::NCW>(p, si, threadIdx.x, &ctl->last);
}

// ---------------------------------------------------------------- head-group tiles
// One CTA per (split, group of kHeadGroup kv heads, row).  A tile is TOK tokens (16 for
// bf16, 32 for FP8) of the row -- of one page when paged -- for the group's kHeadGroup
// heads: one TMA box of TOK rows x kHeadGroup heads (16 KB) per K and V, laid out
// [head][line][row][128 B] -- the same shared-memory layout as kHeadGroup page boxes of
// TOK rows, so the consumer's addressing is unchanged: consumer warp w reads tile rows
// TOK w .. TOK w + TOK - 1, which are head g0 + w's TOK tokens.  Each warp therefore
// sees every token of its own head in the split and writes that head's partial itself;
// no cross-warp merge.
template <class SH>
__global__ void __launch_bounds__(SH::THREADS, 2)
    fd_partial_heads_kernel(const __grid_constant__ CUtensorMap tk,
                            const __grid_constant__ CUtensorMap tv,
                            const __grid_constant__ Params p) {
  // Tokens of one head in a tile: 16 (bf16) or 32 (FP8), so that the box of kHeadGroup
  // heads is kTileBytes -- and exactly one consumer warp's rows of the tile.
  constexpr int STAGES = SH::STAGES, TOK = SH::ROWS_PER_WARP;
  static_assert(SH::NCW == kHeadGroup && TOK * kHeadGroup == SH::TT && !SH::WIDE && !SH::F32,
                "one head's tokens per consumer warp");
  // (Not with 16 query rows per kv head: there its registers would spill.)
  if constexpr (SH::G <= 8) {
    if (threadIdx.x == SH::NCW * 32) {
      if (p.block_table != nullptr)
        prefetch_first_pages<TOK>(p, &tk, &tv, kPrefetchHeadTiles, (int)blockIdx.y * kHeadGroup);
      else
        prefetch_first_tiles<TOK>(p, &tk, &tv, kPrefetchHeadTiles, (int)blockIdx.y * kHeadGroup);
    }
  }
  pdl_wait();                       // inputs of this step are visible
  SplitInfo si = split_info<TOK>(p);
  si.g = blockIdx.y * kHeadGroup;                 // first kv head of the group
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  auto* ctl = reinterpret_cast<PipeCtl<STAGES>*>(stages + SH::RING_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (si.n_tiles == 0) {            // empty split for every head of the group
    for (int i = threadIdx.x; i < kHeadGroup * p.n_rows; i += blockDim.x)
      put_empty_row<Consumer<SH>::direct_ok()>(p, si.b, si.g + i / p.n_rows, i % p.n_rows, si.split);
    pdl_trigger();
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_addr(&ctl->full[s]), 1);
      mbar_init(smem_addr(&ctl->empty[s]), SH::NCW);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == SH::NCW) {            // producer: one 16-row box of the group per K and V
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
    produce_tiles<TOK, STAGES, kHeadGroup>(p, si, &tk, &tv, stages, ctl, lane);
    pdl_trigger();
    return;
  }

  const int g = si.g + warp;        // this warp's kv head
  Consumer<SH> c;
  c.start(p, si.b, g, si.L, lane);
  const int r0 = warp * TOK;
  bool aborted = false;
  for (int n = 0; n < si.n_tiles; ++n) {
    const int stage = n % STAGES;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_addr(&ctl->full[stage]), (n / STAGES) & 1);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        ctl->abort = 1;
        atomicOr(p.flags, kDevFlagTimeout);
      }
      aborted = true;
      break;
    }
    uint8_t* kt = stages + (size_t)stage * 2 * kTileBytes;
    // Row r0 + i of the tile is token t0 + i of head g: pass the row-0 token as t0 - r0.
    const int64_t t0 = si.T0 + (int64_t)n * TOK;
    c.tile(p, kt, kt + kTileBytes, t0 - r0, si.lo, si.hi, ctl->bad[stage], warp, lane,
           (uint32_t)p.log2_box, false);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl->empty[stage]));
  }
  pdl_trigger();
  if (aborted || *reinterpret_cast<volatile int32_t*>(&ctl->abort)) {
    if (lane < p.n_rows) put_empty_row<Consumer<SH>::direct_ok()>(p, si.b, g, lane, si.split);
    return;
  }
  c.store_own(p, si.b, g, si.split, lane);
}

// ---------------------------------------------------------------- persistent schedule
// Two CTAs per SM for the whole pass.  The producer warp takes (split, kv head, row)
// items from a queue in the workspace and streams their tiles back to back; the
// consumers follow the tiles' metadata, restart their state at an item's first tile and,
// at its last, merge the four warps' states in that tile's stage before releasing it.
// No per-item CTA launch, pipeline fill or partial last wave.
template <class SH>
__global__ void __launch_bounds__(SH::THREADS, 2)
    fd_partial_persist_kernel(const __grid_constant__ CUtensorMap tk,
                              const __grid_constant__ CUtensorMap tv,
                              const __grid_constant__ Params p) {
  constexpr int G = SH::G, TT = SH::TT, STAGES = SH::STAGES;
  // (Not with 16 query rows per kv head, whose registers are at the cap.)
  if constexpr (G <= 8) {
    if (threadIdx.x == SH::NCW * 32) prefetch_first_item<TT, 1>(p, &tk, &tv, kPrefetchTiles);
  }
  pdl_wait();                       // inputs of this step are visible
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  auto* ctl = reinterpret_cast<PersistCtl<STAGES>*>(stages + SH::RING_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_addr(&ctl->full[s]), 1);
      mbar_init(smem_addr(&ctl->empty[s]), SH::NCW);
    }
    for (int i = 0; i < 3; ++i) mbar_init(smem_addr(&ctl->epi[i]), SH::NCW);
    ctl->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == SH::NCW) {
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
    produce_items<TT, STAGES, (G <= 8)>(p, &tk, &tv, stages, ctl, lane);
    pdl_trigger();
    return;
  }

  // The consumer warps meet around each item's epilogue on mbarriers with bounded waits
  // rather than a hardware barrier: a warp that gave up on a stalled stage must not
  // leave the others blocked.
  uint32_t epi_phase = 0;
  auto meet = [&](int which) -> bool {
    __syncwarp();
    int ok = 1;
    if (lane == 0) {
      mbar_arrive(smem_addr(&ctl->epi[which]));
      ok = mbar_wait(smem_addr(&ctl->epi[which]), epi_phase & 1);
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  auto give_up = [&]() {
    if (lane == 0) {
      ctl->abort = 1;
      atomicOr(p.flags, kDevFlagTimeout);
    }
  };

  Consumer<SH> c;
  const bool multi_page = p.page_size > 0 && p.page_size < TT;
  const uint32_t lb = (uint32_t)p.log2_box;
  for (int n = 0;; ++n) {
    const int stage = n % STAGES;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_addr(&ctl->full[stage]), (n / STAGES) & 1);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      give_up();
      break;
    }
    const TileMeta mt = ctl->meta[stage];
    if (mt.flags & kMetaDone) break;
    if (mt.flags & kMetaFirst) c.start(p, mt.b, mt.g, mt.L, lane);
    uint8_t* kt = stages + (size_t)stage * 2 * kTileBytes;
    c.tile(p, kt, kt + kTileBytes, mt.t0, mt.lo, mt.hi, mt.bad, warp, lane, lb, multi_page);
    if (mt.flags & kMetaLast) {
      // The stage becomes the merge scratch macc [NCW][G][D] once every warp is done
      // with its K/V rows; mm, ml [NCW][G] live in the control block.
      if (!meet(0)) {
        give_up();
        break;
      }
      float* macc = reinterpret_cast<float*>(kt);
      c.store(p, macc, ctl->mm, ctl->ml, warp, lane);
      if (!meet(1)) {
        give_up();
        break;
      }
      SplitInfo si{};
      si.b = mt.b;
      si.g = mt.g;
      si.split = mt.split;
      if (!merge_warps_and_store<G, SH::D, SH::NCW, (G <= 8)>(p, si, macc, ctl->mm, ctl->ml, threadIdx.x,
                                                    [&] { return meet(2); })) {
        give_up();
        break;
      }
      ++epi_phase;
      // Generic-proxy use of the stage ends before its next TMA fill.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl->empty[stage]));
  }
  pdl_trigger();
}

// ---------------------------------------------------------------- persistent head groups
// The persistent schedule over head-group tiles: items are (split, group of kHeadGroup
// kv heads, row), taken from the queue as above, and each tile is one box of TOK tokens
// x kHeadGroup heads.  Consumer warp w owns head g0 + w of every item, as in the
// head-group kernel: it restarts its state at an item's first tile and writes its head's
// partial at the item's last, with no cross-warp merge -- so the warps never wait for one
// another, and the producer streams the next item while they finish the last one.  The
// per-item arithmetic is the head-group kernel's, bit for bit.
template <class SH>
__global__ void __launch_bounds__(SH::THREADS, 2)
    fd_partial_heads_persist_kernel(const __grid_constant__ CUtensorMap tk,
                                    const __grid_constant__ CUtensorMap tv,
                                    const __grid_constant__ Params p) {
  constexpr int STAGES = SH::STAGES, TOK = SH::ROWS_PER_WARP;
  static_assert(SH::NCW == kHeadGroup && TOK * kHeadGroup == SH::TT && !SH::WIDE && !SH::F32,
                "one head's tokens per consumer warp");
  if constexpr (SH::G <= 8) {
    if (threadIdx.x == SH::NCW * 32)
      prefetch_first_item<TOK, kHeadGroup>(p, &tk, &tv, kPrefetchHeadTiles);
  }
  pdl_wait();                       // inputs of this step are visible
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  auto* ctl = reinterpret_cast<PersistCtl<STAGES>*>(stages + SH::RING_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_addr(&ctl->full[s]), 1);
      mbar_init(smem_addr(&ctl->empty[s]), SH::NCW);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == SH::NCW) {
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
    produce_items<TOK, STAGES, Consumer<SH>::direct_ok(), kHeadGroup>(p, &tk, &tv, stages, ctl, lane);
    pdl_trigger();
    return;
  }

  Consumer<SH> c;
  const int r0 = warp * TOK;
  const uint32_t lb = (uint32_t)p.log2_box;
  bool open = false;                // an item started and not yet written
  TileMeta mt{};
  for (int n = 0;; ++n) {
    const int stage = n % STAGES;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_addr(&ctl->full[stage]), (n / STAGES) & 1);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        ctl->abort = 1;
        atomicOr(p.flags, kDevFlagTimeout);
      }
      break;
    }
    mt = ctl->meta[stage];
    if (mt.flags & kMetaDone) break;
    const int g = mt.g + warp;      // this warp's kv head
    if (mt.flags & kMetaFirst) {
      c.start(p, mt.b, g, mt.L, lane);
      open = true;
    }
    uint8_t* kt = stages + (size_t)stage * 2 * kTileBytes;
    // Row r0 + i of the tile is token t0 + i of head g: pass the row-0 token as t0 - r0.
    c.tile(p, kt, kt + kTileBytes, mt.t0 - r0, mt.lo, mt.hi, mt.bad, warp, lane, lb, false);
    if (mt.flags & kMetaLast) {
      c.store_own(p, mt.b, g, mt.split, lane);
      open = false;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl->empty[stage]));
  }
  // An item left half done by a wait that ran out: weight 0 for this warp's head.
  if (open && lane < p.n_rows)
    put_empty_row<Consumer<SH>::direct_ok()>(p, mt.b, mt.g + warp, lane, mt.split);
  pdl_trigger();
}

// ---------------------------------------------------------------- persistent wide groups
// The persistent schedule over the wide kernel's items (split, kv head, row) of 17 to 32
// query rows: consumer warp w keeps rows 8 w .. 8 w + 7 of every item over each whole
// tile, restarts them at an item's first tile and writes their partial at its last, so
// the warps never wait for one another and the producer streams the next item while
// they finish.  Per item, the arithmetic is the wide kernel's, bit for bit.
template <class SH>
__global__ void __launch_bounds__(SH::THREADS, 2)
    fd_partial_wide_persist_kernel(const __grid_constant__ CUtensorMap tk,
                                   const __grid_constant__ CUtensorMap tv,
                                   const __grid_constant__ Params p) {
  constexpr int TT = SH::TT, STAGES = SH::STAGES;
  static_assert(SH::WIDE && SH::PERSIST && SH::G == 8, "wide groups of up to 32 rows");
  if (threadIdx.x == SH::NCW * 32) prefetch_first_item<TT, 1>(p, &tk, &tv, kPrefetchTiles);
  pdl_wait();                       // inputs of this step are visible
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  auto* ctl = reinterpret_cast<PersistCtl<STAGES>*>(stages + SH::RING_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_addr(&ctl->full[s]), 1);
      mbar_init(smem_addr(&ctl->empty[s]), SH::NCW);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == SH::NCW) {
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
    produce_items<TT, STAGES, Consumer<SH>::direct_ok(), 1>(p, &tk, &tv, stages, ctl, lane);
    pdl_trigger();
    return;
  }

  Consumer<SH> c;
  const bool multi_page = p.page_size > 0 && p.page_size < TT;
  const uint32_t lb = (uint32_t)p.log2_box;
  bool open = false;                // an item started and not yet written
  TileMeta mt{};
  for (int n = 0;; ++n) {
    const int stage = n % STAGES;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_addr(&ctl->full[stage]), (n / STAGES) & 1);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        ctl->abort = 1;
        atomicOr(p.flags, kDevFlagTimeout);
      }
      break;
    }
    mt = ctl->meta[stage];
    if (mt.flags & kMetaDone) break;
    if (mt.flags & kMetaFirst) {
      c.start(p, mt.b, mt.g, mt.L, lane, warp * SH::G);
      open = true;
    }
    uint8_t* kt = stages + (size_t)stage * 2 * kTileBytes;
    c.tile(p, kt, kt + kTileBytes, mt.t0, mt.lo, mt.hi, mt.bad, warp, lane, lb, multi_page);
    if (mt.flags & kMetaLast) {
      c.store_own(p, mt.b, mt.g, mt.split, lane);
      open = false;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl->empty[stage]));
  }
  // An item left half done by a wait that ran out: weight 0 for this warp's rows.
  if (open) {
    const int h = warp * SH::G + lane;
    if (lane < SH::G && h < p.n_rows) put_empty_row<Consumer<SH>::direct_ok()>(p, mt.b, mt.g, h, mt.split);
  }
  pdl_trigger();
}

template <class SH>
cudaError_t launch_mma(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t stream) {
  cudaError_t e;
  if constexpr (SH::PERSIST && SH::WIDE) {
    auto kernel = fd_partial_wide_persist_kernel<SH>;
    static SmemOptIn opt_in;
    e = opt_in.apply(kernel, (int)SH::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int64_t items = (int64_t)p.S * p.Hkv * p.B;
    const unsigned grid = (unsigned)(items < 2 * sms ? items : 2 * sms);
    e = launch_partial_kernel(kernel, dim3(grid), SH::THREADS, SH::SMEM_BYTES, stream, tk, tv, p);
  } else if constexpr (SH::PERSIST) {
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    if (p.head_group) {
      if constexpr (SH::D == 128) {
        auto kernel = fd_partial_heads_persist_kernel<SH>;
        static SmemOptIn opt_in;
        e = opt_in.apply(kernel, (int)SH::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        const int64_t items = (int64_t)p.S * (p.Hkv / kHeadGroup) * p.B;
        const unsigned grid = (unsigned)(items < 2 * sms ? items : 2 * sms);
        e = launch_partial_kernel(kernel, dim3(grid), SH::THREADS, SH::SMEM_BYTES, stream, tk,
                                  tv, p);
      } else {
        return cudaErrorInvalidValue;   // the host enables head groups for d = 128 only
      }
    } else {
      auto kernel = fd_partial_persist_kernel<SH>;
      static SmemOptIn opt_in;
      e = opt_in.apply(kernel, (int)SH::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      const int64_t items = (int64_t)p.S * p.Hkv * p.B;
      const unsigned grid = (unsigned)(items < 2 * sms ? items : 2 * sms);
      e = launch_partial_kernel(kernel, dim3(grid), SH::THREADS, SH::SMEM_BYTES, stream, tk, tv,
                                p);
    }
  } else if constexpr (SH::WIDE) {
    auto kernel = fd_partial_wide_kernel<SH>;
    static SmemOptIn opt_in;
    e = opt_in.apply(kernel, (int)SH::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)p.S, (unsigned)p.Hkv, (unsigned)p.B);
    e = launch_partial_kernel(kernel, grid, SH::THREADS, SH::SMEM_BYTES, stream, tk, tv, p);
  } else if (p.head_group) {
    if constexpr (SH::D == 128 && !SH::F32) {
      auto kernel = fd_partial_heads_kernel<SH>;
      static SmemOptIn opt_in;
      e = opt_in.apply(kernel, (int)SH::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      dim3 grid((unsigned)p.S, (unsigned)(p.Hkv / kHeadGroup), (unsigned)p.B);
      Params q = p;
      q.wave = 2 * sm_count();      // two CTAs per SM
      e = launch_partial_kernel(kernel, grid, SH::THREADS, SH::SMEM_BYTES, stream, tk, tv, q);
    } else {
      return cudaErrorInvalidValue;   // the host enables head groups for d = 128 only
    }
  } else {
    auto kernel = fd_partial_mma_kernel<SH>;
    static SmemOptIn opt_in;
    e = opt_in.apply(kernel, (int)SH::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)p.S, (unsigned)p.Hkv, (unsigned)p.B);
    Params q = p;
    q.wave = 2 * sm_count();        // two CTAs per SM
    e = launch_partial_kernel(kernel, grid, SH::THREADS, SH::SMEM_BYTES, stream, tk, tv, q);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, bool KV8, bool PERSIST>
cudaError_t dispatch_g(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t stream) {
  switch (rows_template(p.n_rows)) {   // query rows per (b, kv head), padded
    case 1: return launch_mma<MmaShape<D, 1, KV8, PERSIST>>(p, tk, tv, stream);
    case 2: return launch_mma<MmaShape<D, 2, KV8, PERSIST>>(p, tk, tv, stream);
    case 4: return launch_mma<MmaShape<D, 4, KV8, PERSIST>>(p, tk, tv, stream);
    case 8: return launch_mma<MmaShape<D, 8, KV8, PERSIST>>(p, tk, tv, stream);
    case 16: return launch_mma<MmaShape<D, 16, KV8, PERSIST>>(p, tk, tv, stream);
    case 32:   // wide groups: four warps of 8 rows (bf16 or FP8 KV)
      return launch_mma<MmaShape<D, 8, KV8, PERSIST, true>>(p, tk, tv, stream);
    case 64:   // four warps of 16 rows
      if constexpr (!KV8 && !PERSIST) return launch_mma<MmaShape<D, 16, false, false, true>>(p, tk, tv, stream);
      else return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
cudaError_t dispatch_f32(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                         cudaStream_t stream) {
  switch (rows_template(p.n_rows)) {
    case 1: return launch_mma<MmaShape<D, 1, false, false, false, true>>(p, tk, tv, stream);
    case 2: return launch_mma<MmaShape<D, 2, false, false, false, true>>(p, tk, tv, stream);
    case 4: return launch_mma<MmaShape<D, 4, false, false, false, true>>(p, tk, tv, stream);
    case 8: return launch_mma<MmaShape<D, 8, false, false, false, true>>(p, tk, tv, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <bool PERSIST>
cudaError_t dispatch_kind(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                          cudaStream_t stream) {
  if (p.in_f32) {   // the host runs f32 inputs here on the grid schedule only
    if constexpr (PERSIST) return cudaErrorInvalidValue;
    else if (p.head_group) return cudaErrorInvalidValue;
    else return p.d == 128 ? dispatch_f32<128>(p, tk, tv, stream)
                           : p.d == 64 ? dispatch_f32<64>(p, tk, tv, stream) : cudaErrorInvalidValue;
  }
  if (p.kv_fp8) return p.d == 128 ? dispatch_g<128, true, PERSIST>(p, tk, tv, stream) : cudaErrorInvalidValue;
  if (p.d == 128) return dispatch_g<128, false, PERSIST>(p, tk, tv, stream);
  if (p.d == 64) return dispatch_g<64, false, PERSIST>(p, tk, tv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

// The kernels launch_partial_mma runs with 16 rows per warp -- head groups, the wide
// kernel for 33 to 64 rows and the persistent schedule -- write partials only (their
// Consumer<SH>::direct_ok() / DIRECT forms); every other instantiation also writes a single
// split's result as the output.
bool mma_writes_direct(const Params& p) {
  const int r = rows_template(p.n_rows);
  if (r == 32) return true;         // wide groups, 8 rows a warp (grid or persistent)
  if (p.head_group || p.persistent) return r <= 8;
  return r != 64;
}

cudaError_t launch_partial_mma(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t stream) {
  return p.persistent ? dispatch_kind<true>(p, tk, tv, stream)
                      : dispatch_kind<false>(p, tk, tv, stream);
}

}  // namespace fd
