// fd_partial_tc.cu -- split-KV partial pass on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory), for groups of up to 64 query rows per
// kv head: multi-token decode on GQA groups (Q query tokens x G heads), or groups of
// 32 and 64 heads.  bf16 inputs, d = 128.
//
// Per tile of TT = 64 tokens of one kv head (the TMA tiles of fd_pipeline.cuh, used as
// the mma operands in place):
//   S[128, TT]  = Q[128, d] . K_tile^T          tcgen05.mma, Q in TMEM, K the tile in
//                                               shared memory, M = 128, N = TT, into TMEM
//   one thread per TMEM lane reads its row of S (tcgen05.ld), masks it, keeps the
//   running max m and sum l, and writes P = bf16(2^(S - m)) back to TMEM (tcgen05.st)
//   O[128, d]  += P[128, TT] . V_tile[TT, d]    tcgen05.mma, P in TMEM, V read from the
//                                               tile as an MN-major operand, O in TMEM
// This is the FlashAttention block update of "AI Infra: math and infra optimisation in
// large models", section 2.6, inside one split of Flash-Decoding (same section, Split-K):
// S = Q K^T per KV block; rescale the running sum and output by exp(m_old - m_new); add
// exp(S - m_new) V.  The running max only moves (and O in TMEM is rescaled) when a
// tile's max exceeds it by more than 8 in base-2 units: every 2^(S - m) then stays at
// most 2^8, and since l and O use the same m throughout, the result is unchanged.
//
// Why: with R query rows per kv head each KV byte feeds R flops, and past 32 rows the
// mma.sync kernels become bound by issue latency and by every warp re-reading the tile
// from shared memory.  Here one thread issues each tile's products as a few large
// instructions that read the tile once, and the other warps only do the softmax.
//
// Warps: 0-7 softmax in two groups of four, 8 the TMA producer, 9 and 10 the issuers of
// the even and odd tiles' score products, 11 the issuer of the output products (one
// thread each).  Group g takes the tiles n = g mod 2 with its own S buffer, P buffer and O
// accumulator, so the two groups' per-tile handoffs (scores ready, P written, product
// done) overlap.  The 128 rows of the products are the R query rows repeated 128 / R
// times (Q is stored that way): TMEM lane L holds query row L mod R, and its thread
// takes the slice L / R of each tile's tokens (TT R / 128 of them), with its own running
// max and sum (P is zero outside the slice).  The 2 x 128 / R partial states of a row
// are merged at the end of the split, like the warps of the mma.sync kernel.  One CTA
// per SM: 6 stages of K + V (192 KB) in shared memory; 512 TMEM columns: S 2 x 64,
// O 2 x 128, Q 64 (128 dims as bf16 pairs), P 2 x 32.  With Q and P in TMEM, shared
// memory carries only the K and V operands (each read once per tile).
#include <cuda_bf16.h>

#include "fd_epilogue.cuh"

namespace fd {
namespace {

constexpr int kTcD = 128;
constexpr int kTcTT = 64;                    // tokens per tile (16 KB of K, 16 KB of V)
// An even number of stages: stage st then only ever holds tiles of parity st % 2, so the
// roles that take one parity of tiles (a softmax group, a score issuer) see every phase
// of the stage's barrier -- a parity wait is only exact for a waiter that never skips one.
constexpr int kTcStages = 6;
static_assert(kTcStages % 2 == 0, "stages hold tiles of one parity");
constexpr int kTcThreads = 384;
constexpr int kTcSoftThreads = 256;          // two groups of four warps
constexpr uint32_t kTcCols = 512;            // TMEM columns:
constexpr uint32_t kTcOCol = 128;            //   S 0..127, O of group g at 128 + 128 g,
constexpr uint32_t kTcQCol = 384;            //   Q (bf16 pairs along d),
constexpr uint32_t kTcPCol = 448;            //   P of group g at 448 + 32 g (bf16 pairs)
// Shared memory, from a 1024-byte aligned base: the ring, then the control block.
constexpr uint32_t kTcCtlOff = kTcStages * 2 * kTileBytes;  // 192 KB

struct TcCtl {
  PipeCtl<kTcStages> pipe;   // TMA ring (empty: released by the output issuer's commit)
  uint64_t s_full[2];        // S buffer b holds a finished Q K^T (tcgen05.commit)
  uint64_t s_free[2];        // the softmax warps have read S buffer b
  uint64_t p_full[2];        // P of tile n (and its zeroed V rows) is in place, n % 2 = b
                             // (two barriers: the softmax may finish tile n + 1 before
                             // the output issuer has seen tile n, and a parity wait must
                             // never be two phases behind its barrier)
  uint64_t pv_done[2];       // the P V product of a tile of parity b has completed
  uint64_t mma_done;         // every product this CTA issued has completed (three issuers)
  uint32_t tmem;             // TMEM base address (tcgen05.alloc)
};
constexpr size_t kTcSmemBytes = 1024 + kTcCtlOff + ((sizeof(TcCtl) + 127) / 128) * 128;
static_assert(kTcSmemBytes <= 227 * 1024, "one CTA per SM");

// ---------------------------------------------------------------- tcgen05 wrappers
__device__ __forceinline__ void tc_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D (TMEM) = A . B (+ D), A in TMEM (lane = row, K packed two bf16 per column).
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      :: "r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(bar) : "memory");
}
// TMEM -> registers: 32 consecutive f32 columns of this thread's lane (a warp reads
// lanes 32 (warp % 4) .. + 31), with the wait inside the same asm statement so that no
// use of the registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// Two 32-column TMEM loads (columns taddr0.., taddr1..) with a single wait.
__device__ __forceinline__ void tc_ld32x2(uint32_t taddr0, uint32_t taddr1, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr0), "r"(taddr1)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Registers -> TMEM (32 columns of the lane), complete before the statement ends.
__device__ __forceinline__ void tc_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;"
      :: "r"(taddr), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
         "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]),
         "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]),
         "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}
// Registers -> TMEM, 32 columns of raw words (bf16 pairs), complete before the statement ends.
__device__ __forceinline__ void tc_st32w(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;"
      :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
         "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
         "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
         "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
// Registers -> TMEM, 16 or 8 columns of packed words, complete before the statement ends.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
      "%10, %11, %12, %13, %14, %15, %16};\n\t"
      "tcgen05.wait::st.sync.aligned;"
      :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
         "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
         "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tc_st8(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n\t"
      "tcgen05.wait::st.sync.aligned;"
      :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory operand descriptor, 128-byte swizzle: start address, leading and stride
// byte offsets (16-byte units), descriptor version 1, layout 2 = SWIZZLE_128B.
//   K-major operand (the K tile: rows of 128 bytes = 64 bf16 along K): stride = 1024
//   (one 8-row swizzle atom to the next along N); the leading offset is not used.  A
//   k-step of 16 elements inside the atom advances the start address by 32 bytes.
//   MN-major operand (the V tile: a row is one token, 128 bytes = 64 dims along N):
//   leading = bytes from one 64-dim slab to the next, stride = 1024 (8 tokens).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lead, uint32_t stride) {
  return (uint64_t)((addr >> 4) & 0x3fffu) | ((uint64_t)((lead >> 4) & 0x3fffu) << 16) |
         ((uint64_t)((stride >> 4) & 0x3fffu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: f32 accumulator, bf16 A and B, A K-major (here A
// is always in TMEM), B K-major (b_mn = 0) or MN-major (1), N >> 3 and M >> 4.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// A bounded wait whose outcome every lane of the warp shares.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(bar, parity);
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void set_abort(const Params& p, TcCtl* ctl) {
  *reinterpret_cast<volatile int32_t*>(&ctl->pipe.abort) = 1;
  atomicOr(p.flags, kDevFlagTimeout);
}
__device__ __forceinline__ bool aborted(TcCtl* ctl) {
  return *reinterpret_cast<volatile int32_t*>(&ctl->pipe.abort) != 0;
}

// ---------------------------------------------------------------- mma issuer
// Probe that may suspend the thread for up to `hint_ns` while the phase is incomplete.
__device__ __forceinline__ bool mbar_probe(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// A bounded wait that also gives up as soon as another role has aborted the split.
__device__ __forceinline__ bool wait_or_abort(TcCtl* ctl, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;     // the common case reads no timer
  const uint64_t t0 = global_ns();
  while (!mbar_probe(bar, parity, 200u)) {
    if (aborted(ctl) || global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// Whether ring slot n (landed) carries the end of the tile sequence rather than a tile.
__device__ __forceinline__ bool tile_done(TcCtl* ctl, int n) {
  return *reinterpret_cast<volatile int32_t*>(&ctl->pipe.done[n % kTcStages]) != 0;
}

// The products are issued by three threads in three warps: two issue the scores
// S(j) = Q K(j)^T of the even and of the odd tiles, each as soon as tile j has landed
// and its S buffer has been read (the softmax of tile j - 2); the third issues the
// products P(n) V(n) of all tiles in order, each as soon as P(n) is in place.  They
// write disjoint TMEM columns and read different operands, so none waits for another's
// instruction stream; a stage is released by the third's commit after P(n) V(n), which
// implies S(n) has completed (the softmax read it before writing P(n)).  Each thread
// finishes by waiting for all of its products.
__device__ void issue_scores(const Params& p, const SplitInfo& si, uint8_t* stages,
                             TcCtl* ctl, uint32_t tmem, int parity) {
  const bool multi_page = p.block_table != nullptr && p.page_size < kTcTT;
  const int box = multi_page ? p.page_size : kTcTT;     // token rows of one TMA box
  const int nbox = kTcTT / box;
  const uint32_t box_bytes = 2u * (uint32_t)box * 128u;  // [line][row][128 B], 2 lines
  const uint32_t id_s = instr_desc(128, box, 0);
  bool ok = true;
  for (int j = parity;; j += 2) {
    if (!wait_or_abort(ctl, smem_addr(&ctl->pipe.full[j % kTcStages]), (j / kTcStages) & 1)) {
      ok = false;
      break;
    }
    if (tile_done(ctl, j)) break;           // no tile j: the sequence has ended
    if (j >= 2 && !wait_or_abort(ctl, smem_addr(&ctl->s_free[j & 1]), ((j >> 1) - 1) & 1)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t kb = smem_addr(stages + (size_t)(j % kTcStages) * 2 * kTileBytes);
    for (int bx = 0; bx < nbox; ++bx) {
#pragma unroll
      for (int ks = 0; ks < kTcD / 16; ++ks) {
        const uint64_t b = smem_desc(kb + bx * box_bytes + (ks >> 2) * (uint32_t)box * 128u +
                                         (ks & 3) * 32u, 0, 1024);
        tc_mma_ts(tmem + (j & 1) * kTcTT + bx * box, tmem + kTcQCol + ks * 8, b, id_s, ks > 0);
      }
    }
    tc_commit(smem_addr(&ctl->s_full[j & 1]));
  }
  if (!ok) set_abort(p, ctl);
  tc_commit(smem_addr(&ctl->mma_done));      // never leave with products in flight
  if (!mbar_wait(smem_addr(&ctl->mma_done), 0)) atomicOr(p.flags, kDevFlagTimeout);
}

__device__ void issue_outputs(const Params& p, const SplitInfo& si, uint8_t* stages,
                              TcCtl* ctl, uint32_t tmem) {
  const bool multi_page = p.block_table != nullptr && p.page_size < kTcTT;
  const int box = multi_page ? p.page_size : kTcTT;
  const uint32_t box_bytes = 2u * (uint32_t)box * 128u;
  const uint32_t id_pv = instr_desc(128, kTcD, 1);
  bool ok = true;
  for (int n = 0;; ++n) {
    if (!wait_or_abort(ctl, smem_addr(&ctl->pipe.full[n % kTcStages]), (n / kTcStages) & 1)) {
      ok = false;
      break;
    }
    if (tile_done(ctl, n)) break;           // no tile n: the sequence has ended
    if (!wait_or_abort(ctl, smem_addr(&ctl->p_full[n & 1]), (n >> 1) & 1)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const int st = n % kTcStages;
    const uint32_t vb = smem_addr(stages + (size_t)st * 2 * kTileBytes + kTileBytes);
    const uint32_t pt = tmem + kTcPCol + (uint32_t)(n & 1) * (kTcTT / 2);
#pragma unroll
    for (int ks = 0; ks < kTcTT / 16; ++ks) {
      const int tok = ks * 16, bx = tok / box, rr = tok % box;
      const uint64_t b = smem_desc(vb + bx * box_bytes + (uint32_t)rr * 128u,
                                   (uint32_t)box * 128u, 1024);
      tc_mma_ts(tmem + kTcOCol + (uint32_t)(n & 1) * kTcD, pt + ks * 8, b, id_pv,
                (n > 1 || ks > 0) ? 1u : 0u);
    }
    tc_commit(smem_addr(&ctl->pv_done[n & 1]));
    tc_commit(smem_addr(&ctl->pipe.empty[st]));
  }
  if (!ok) set_abort(p, ctl);
  tc_commit(smem_addr(&ctl->mma_done));
  if (!mbar_wait(smem_addr(&ctl->mma_done), 0)) atomicOr(p.flags, kDevFlagTimeout);
}

// ---------------------------------------------------------------- softmax warps
// Thread t (0..255): group g = t / 128 takes tiles n = g mod 2; within it, TMEM lane
// tg = t mod 128 holds query row h = tg mod R and the token slice tg / R of each tile.
// Returns false if a bounded wait gave up.
template <int R>
__device__ bool softmax_rows(const Params& p, const SplitInfo& si, uint8_t* stages,
                             TcCtl* ctl, uint32_t tmem, int t, float& m_out, float& l_out,
                             int& n_total) {
  constexpr int SLICE = kTcTT * R / 128;             // tokens of a tile per lane: 32 or 16
  const int grp = t >> 7, tg = t & 127;
  const int warp = tg >> 5, lane = t & 31;
  const int h = tg % R, slice = tg / R;
  const int64_t kb = key_bound(p, si.L, h);          // causal bound of row h
  const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
  const bool multi_page = p.block_table != nullptr && p.page_size < kTcTT;
  const uint32_t lb = (uint32_t)p.log2_box;
  const float sl2 = p.scale_log2;
  const int j0 = slice * SLICE;                      // first token of the slice in a tile
  const uint32_t ocol = kTcOCol + (uint32_t)grp * kTcD;
  const uint32_t pcol = kTcPCol + (uint32_t)grp * (kTcTT / 2) + (uint32_t)(j0 / 2);
  float m = kNegInf, l = 0.f;
  int last = -1;                                     // the group's last tile
  for (int n = grp;; n += 2) {
    const int st = n % kTcStages;
    // The tile has landed (for its range and page-validity bits) and its scores are
    // complete -- or the slot carries the end of the sequence.
    if (!warp_wait(smem_addr(&ctl->pipe.full[st]), (n / kTcStages) & 1, lane)) return false;
    if (tile_done(ctl, n)) {
      n_total = *reinterpret_cast<volatile int32_t*>(&ctl->pipe.n_total);
      break;
    }
    last = n;
    if (!warp_wait(smem_addr(&ctl->s_full[n & 1]), (n >> 1) & 1, lane)) return false;
    tc_fence_after();
    float s[SLICE];
    if constexpr (SLICE == 32) tc_ld32(tl + (n & 1) * kTcTT + j0, s);
    else tc_ld16(tl + (n & 1) * kTcTT + j0, s);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl->s_free[n & 1]));

    // The tile's first token and the valid range of the split it belongs to (its own
    // split, or one it took from, with tail sharing).
    const int64_t t0 = ctl->pipe.t0[st], lo = ctl->pipe.lo[st], hi = ctl->pipe.hi[st];
    const uint32_t bad = ctl->pipe.bad[st];
    const bool clean = t0 >= lo && t0 + kTcTT <= hi && bad == 0;
    float mt = kNegInf;
    if (clean && t0 + j0 + SLICE <= kb) {
#pragma unroll
      for (int j = 0; j < SLICE; ++j) {
        s[j] *= sl2;
        mt = fmaxf(mt, s[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < SLICE; ++j) {
        const int64_t tok = t0 + j0 + j;
        const int pslot = multi_page ? ((j0 + j) >> p.log2_page) : 0;
        const bool valid = tok >= lo && tok < hi && !((bad >> pslot) & 1u) && tok < kb;
        s[j] = valid ? s[j] * sl2 : kNegInf;
        mt = fmaxf(mt, s[j]);
      }
    }
    const float mn = fmaxf(m, mt);
    const bool resc = n > 1 && m != kNegInf && mn > m + 8.f;
    const float mu = (m == kNegInf || resc) ? mn : m;
    const float c = resc ? ex2(m - mn) : 1.f;
    float sum = 0.f;
    uint32_t pk[SLICE / 2];
#pragma unroll
    for (int j = 0; j < SLICE / 2; ++j) {
      const float p0 = s[2 * j] == kNegInf ? 0.f : ex2(s[2 * j] - mu);
      const float p1 = s[2 * j + 1] == kNegInf ? 0.f : ex2(s[2 * j + 1] - mu);
      sum += p0 + p1;
      pk[j] = pack_bf16(p0, p1);
    }
    l = l * c + sum;
    m = mu;

    // The group's previous product (tile n - 2) has completed: its P buffer is free and
    // its O stable (tile n's product is not issued before this warp arrives on p_full).
    if (n >= 2 && !warp_wait(smem_addr(&ctl->pv_done[n & 1]), ((n >> 1) - 1) & 1, lane))
      return false;
    tc_fence_after();
    if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
      for (int q = 0; q < kTcD / 32; ++q) {
        float o[32];
        tc_ld32(tl + ocol + q * 32, o);
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] *= c;
        tc_st32(tl + ocol + q * 32, o);
      }
    }
    // This lane's slice of its P row, into the group's P columns in TMEM (the rest of
    // the row stays zero).
    if constexpr (SLICE == 32) tc_st16(tl + pcol, pk);
    else tc_st8(tl + pcol, pk);
    // Boundary tile: the V rows of tokens outside [lo, hi) or on an invalid page may hold
    // stale values (NaN), and 0 * NaN would poison the product: zero them.
    if (!clean && tg < kTcTT) {
      const int64_t tok = t0 + tg;
      const int pslot = multi_page ? (tg >> p.log2_page) : 0;
      if (!(tok >= lo && tok < hi && !((bad >> pslot) & 1u))) {
        uint8_t* vt = stages + (size_t)st * 2 * kTileBytes + kTileBytes;
#pragma unroll
        for (int c16 = 0; c16 < kTcD * 2 / 16; ++c16)
          *reinterpret_cast<uint4*>(vt + tile_chunk<2>((uint32_t)tg, (uint32_t)c16, lb)) =
              make_uint4(0, 0, 0, 0);
      }
    }
    fence_proxy_async_smem();       // P and V stores -> the tensor core's reads
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl->p_full[n & 1]));   // one per softmax warp
  }
  if (last >= 0 && !warp_wait(smem_addr(&ctl->pv_done[grp]), (last >> 1) & 1, lane))
    return false;
  m_out = m;
  l_out = l;
  return true;
}

// Epilogue scratch in the ring.  When a softmax group has seen the product of its last
// tile, every product up to that tile has completed (one issuing thread, in order) and
// no copy is left to land: the only stage still in use is the one holding the split's
// last tile, which the other group may still be working on.  So the scratch avoids that
// stage: partial state q (R rows x D floats, 32 KB for R = 64, 16 KB for R = 32) sits in
// stage (last + 1 + q / PER) mod STAGES, PER = 32 KB / its size, and the per-state
// statistics in stage (last + 5) mod STAGES -- 5 of the 6 stages, none of them `last`.
// A group can then write its states as soon as it is done, while the other finishes.
template <int R>
__device__ __forceinline__ float* o_state(uint8_t* stages, int last_stage, int q) {
  constexpr int PER = 64 / R;                        // states per 32 KB stage
  const int st = (last_stage + 1 + q / PER) % kTcStages;
  return reinterpret_cast<float*>(stages + (size_t)st * 2 * kTileBytes +
                                  (size_t)(q % PER) * R * kTcD * sizeof(float));
}
__device__ __forceinline__ float* o_stats(uint8_t* stages, int last_stage) {
  return reinterpret_cast<float*>(stages + (size_t)((last_stage + 5) % kTcStages) * 2 * kTileBytes);
}
// Float offset of dims 4 c4 .. 4 c4 + 3 of query row h inside one state's R x D block.
// Within each 128-byte segment of a row the 16-byte chunks are XOR-swizzled by h mod 8:
// 32 lanes writing the same dims of 32 consecutive rows then cover all 8 chunk
// positions (4 wavefronts per 512 bytes, no bank conflict), and a warp reading the 32
// chunks of one row is conflict-free as well.
__device__ __forceinline__ int o_index(int h, int c4) {
  return h * kTcD + (((c4 & ~7) | ((c4 & 7) ^ (h & 7))) << 2);
}
static_assert(kTcStages == 6, "the epilogue scratch takes 5 of 6 stages");

template <int R>
__global__ void __launch_bounds__(kTcThreads, 1)
    fd_partial_tc_kernel(const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv,
                         const __grid_constant__ Params p) {
  static_assert(R == 32 || R == 64, "32 or 64 query rows");
  constexpr int DUP = 128 / R;      // token slices (copies of each query row) per group
  constexpr int NPART = 2 * DUP;    // partial states per query row
  // The first ring's worth of tiles into L2 before the wait (prefetch_first_tiles;
  // measured best at the ring depth: 6 tiles 86.5 us, 8 tiles 86.8 us, none 88.9 us at
  // 8 query tokens on the 128K GQA workload).
  // Contiguous caches only: with 64-token pages the page-id prefetch measured slower on
  // this kernel (97.8 against 95.9 us, 4 query tokens on the 128K GQA workload).
  if (threadIdx.x == 8 * 32) prefetch_first_tiles<kTcTT>(p, &tk, &tv, kTcStages, (int)blockIdx.y);
  pdl_wait();                       // inputs of this step are visible
  const SplitInfo si = split_info<kTcTT>(p);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stages = base;
  auto* ctl = reinterpret_cast<TcCtl*>(base + kTcCtlOff);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  if (si.n_tiles == 0) {            // empty split: weight 0 in the merge, nothing to load
    write_empty_split(p, si, t);
    pdl_trigger();
    if (p.counters != nullptr && warp < 8) arrive_and_merge<kTcD, 8>(p, si, t, &ctl->pipe.last);
    return;
  }

  if (t == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(smem_addr(&ctl->pipe.full[s]), 1);
      mbar_init(smem_addr(&ctl->pipe.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&ctl->s_full[b]), 1);
      mbar_init(smem_addr(&ctl->s_free[b]), 4);
      mbar_init(smem_addr(&ctl->pv_done[b]), 1);
      mbar_init(smem_addr(&ctl->p_full[b]), 4);     // the four warps of group b
    }
    mbar_init(smem_addr(&ctl->mma_done), 3);
    ctl->pipe.abort = 0;
    ctl->pipe.n_total = 0;
    fence_mbar_init();
  }
  __syncthreads();                  // barriers initialised

  float m = kNegInf, l = 0.f;
  int n_total = 0;                  // tiles this CTA streamed (softmax warps)
  if (warp == 8) {                  // ---------------- TMA producer, from the start: the
    prefetch_tensormap(&tk);        // first tiles load while the other warps set up
    prefetch_tensormap(&tv);
    produce_tiles_shared<kTcTT, kTcStages>(p, si, &tk, &tv, stages, &ctl->pipe, lane,
                                           p.tail_share != 0);
  } else {
    // Set-up of the MMA operands (every warp but the producer): tensor memory, Q and the
    // zeroed P columns.
    if (warp == 0) {
      tc_alloc(smem_addr(&ctl->tmem), kTcCols);
      tc_relinquish();
    }
    tc_fence_before();
    named_bar_sync(2, kTcThreads - 32);
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    if (warp < 8) {
      // Lane L = t mod 128 of TMEM: group 0 writes its Q row (query row L mod R, as bf16
      // pairs along d; rows past the group are zero), each group zeroes its P columns
      // (each lane later writes only its slice of them).
      const int L = t & 127;
      const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      if (t < 128) {
        const int h = L % R;
        const bool live = h < p.n_rows;
        const uint4* qrow = reinterpret_cast<const uint4*>(
            reinterpret_cast<const __nv_bfloat16*>(p.q) + q_offset(p, si.b, si.g, live ? h : 0));
        uint32_t qw[kTcD / 2];                         // the row: 16 loads of 16 bytes
#pragma unroll
        for (int c = 0; c < kTcD / 8; ++c) {
          const uint4 x = live ? qrow[c] : make_uint4(0, 0, 0, 0);
          qw[4 * c] = x.x;
          qw[4 * c + 1] = x.y;
          qw[4 * c + 2] = x.z;
          qw[4 * c + 3] = x.w;
        }
        tc_st32w(tl + kTcQCol, qw);
        tc_st32w(tl + kTcQCol + 32, qw + 32);
      }
      float z[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) z[c] = 0.f;
      tc_st32(tl + kTcPCol + (uint32_t)(t >> 7) * (kTcTT / 2), z);
    }
    tc_fence_before();
    named_bar_sync(2, kTcThreads - 32);
    tc_fence_after();

    if (warp == 9 || warp == 10) {    // ---------- score products, even / odd tiles
      if (lane == 0) issue_scores(p, si, stages, ctl, tmem, warp - 9);
      __syncwarp();
    } else if (warp == 11) {          // ---------------- output products
      if (lane == 0) issue_outputs(p, si, stages, ctl, tmem);
      __syncwarp();
    } else {                          // ---------------- softmax
      if (!softmax_rows<R>(p, si, stages, ctl, tmem, t, m, l, n_total) && lane == 0)
        set_abort(p, ctl);
    }
  }
  pdl_trigger();

  if (warp < 8) {
    // Split epilogue of the softmax warps.  Each group writes its partial states (O from
    // tensor memory, m, l) into the scratch as soon as it has seen its last product (see
    // o_state), then all 256 threads merge them.
    const int h = t % R, part = t / R, grp = t >> 7;
    const int last_stage = (max(n_total, 1) - 1) % kTcStages;
    float* stats = o_stats(stages, last_stage);
    float* mm = stats;                                       // [NPART][R]: m, then weights
    float* ml = mm + kTcSoftThreads;                         // [NPART][R]: l
    float* lrow = ml + kTcSoftThreads;                       // [R]: the row's merged sum
    if (!aborted(ctl)) {
      // Partial state t: group t / 128, slice (t mod 128) / R, row t mod R.  A group
      // without tiles (a one-tile split) has an O that was never written: it
      // contributes zeros with weight 0.
      tc_fence_after();
      const uint32_t tl = ctl->tmem + ((uint32_t)((warp & 3) * 32) << 16) + kTcOCol +
                          (uint32_t)grp * kTcD;
      const bool has = grp < n_total;
      float* mine = o_state<R>(stages, last_stage, part);
#pragma unroll 1
      for (int q = 0; q < 2; ++q) {
        float o[64];
        if (has) {
          tc_ld32x2(tl + q * 64, tl + q * 64 + 32, o);
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j) o[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 64; j += 4)
          *reinterpret_cast<float4*>(mine + o_index(h, q * 16 + j / 4)) =
              make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
      }
      mm[t] = m;
      ml[t] = l;
    }
    tc_fence_before();
    named_bar_sync(1, kTcSoftThreads);
    const bool bad = aborted(ctl);
    if (bad) {
      write_empty_split(p, si, t);
    } else {
      // Weights of a row's NPART partial states, merged as the warps of the mma.sync
      // kernel are (M = max m, c = 2^(m - M), L = sum c l, O = sum c O_part / L).
      if (t < p.n_rows) {
        float M = kNegInf;
#pragma unroll
        for (int q = 0; q < NPART; ++q) M = fmaxf(M, mm[q * R + t]);
        float c[NPART], L = 0.f;
#pragma unroll
        for (int q = 0; q < NPART; ++q) {
          const float mq = mm[q * R + t];
          c[q] = (M == kNegInf || mq == kNegInf) ? 0.f : ex2(mq - M);
          L = fmaf(ml[q * R + t], c[q], L);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int q = 0; q < NPART; ++q) mm[q * R + t] = c[q] * inv;
        lrow[t] = L;
        put_lse(p, si.b, si.g, t, si.split,
                L > 0.f ? (M + lg2_approx(L)) * 0.6931471805599453f : kNegInf);
      }
      named_bar_sync(1, kTcSoftThreads);
      // All 256 threads write O_i: thread t takes dims 4 (t mod 32) .. + 3 of the rows
      // t / 32 + 8 k.  Row rho is query token rho / G of head g G + rho mod G (G a power
      // of two).
      const int c4 = t & 31;
      const int lgG = 31 - __clz(p.G);
      const int64_t ostride = (int64_t)p.S * kTcD;
      float* obase = p.o_part + (int64_t)si.split * kTcD + c4 * 4;
#pragma unroll
      for (int k = 0; k < R / 8; ++k) {
        const int hr = (t >> 5) + 8 * k;
        if (hr >= p.n_rows) continue;
        const bool live = lrow[hr] > 0.f;
        if (!live && !p.direct) continue;           // no key in the split: no O_i
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live) {
#pragma unroll
          for (int q = 0; q < NPART; ++q) {
            const float f = mm[q * R + hr];
            const float4 a = *reinterpret_cast<const float4*>(
                o_state<R>(stages, last_stage, q) + o_index(hr, c4));
            acc.x = fmaf(a.x, f, acc.x);
            acc.y = fmaf(a.y, f, acc.y);
            acc.z = fmaf(a.z, f, acc.z);
            acc.w = fmaf(a.w, f, acc.w);
          }
        }
        if (p.direct) {
          put_out4(p, si.b, si.g, hr, c4 * 4, acc);
        } else {
          const int64_t row = ((int64_t)si.b * p.Q + (hr >> lgG)) * p.Hq +
                              (int64_t)si.g * p.G + (hr & (p.G - 1));
          *reinterpret_cast<float4*>(obase + row * ostride) = acc;
        }
      }
    }
    if (p.counters != nullptr) arrive_and_merge<kTcD, 8>(p, si, t, &ctl->pipe.last);
  }
  tc_fence_before();
  __syncthreads();                  // every role done; every product complete
  if (warp == 0) {
    tc_fence_after();
    tc_dealloc(ctl->tmem, kTcCols);
  }
}

template <int R>
cudaError_t launch_tc(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                      cudaStream_t stream) {
  auto kernel = fd_partial_tc_kernel<R>;
  static SmemOptIn opt_in;          // set once per device
  cudaError_t e = opt_in.apply(kernel, (int)kTcSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.S, (unsigned)p.Hkv, (unsigned)p.B);
  Params q = p;
  q.wave = sm_count();              // one CTA per SM
  e = launch_partial_kernel(kernel, grid, kTcThreads, kTcSmemBytes, stream, tk, tv, q);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool partial_tc_supported(const Params& p) {
  return p.d == kTcD && !p.kv_fp8 && !p.in_f32 && p.n_rows >= 1 && p.n_rows <= 64 &&
         p.head_group == 0 && !p.persistent &&
         (p.block_table == nullptr || p.page_size >= 16);
}

cudaError_t launch_partial_tc(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              cudaStream_t stream) {
  if (!partial_tc_supported(p)) return cudaErrorInvalidValue;
  return p.n_rows <= 32 ? launch_tc<32>(p, tk, tv, stream) : launch_tc<64>(p, tk, tv, stream);
}

}  // namespace fd
