// fd_planner.cu -- how many KV splits a decode step should use (host code only).
//
// "2kiu.com/news/6053916", section "the split count is a cost account": more splits
// expose more independent work, but every split adds a partial result, a share of the
// merge, and a start-up cost; on short contexts they can cost more than they return,
// and the choice should follow batch, context, head dim and device.  Both planners
// below work in those terms for this library's kernels, where one CTA streams one split
// of one (b, kv head) pair and two CTAs fit on an SM.
//
// fd_num_splits_heuristic knows only the capacity L_cap (no lengths), so it plans for
// full rows: every (b, kv head, split) CTA then has the same work, and the best split
// count keeps all of them in ONE wave of resident CTAs (a second, partial wave leaves
// most SMs idle at the end) while making split_len a multiple of the tile (a split that
// ends mid-tile makes two CTAs load the same boundary tile).
//
// fd_num_splits_for_lengths knows every row's length (on the host), so ragged batches
// can be planned: it simulates the launch -- CTAs start in launch order as slots free
// up; the running CTAs share an aggregate bandwidth that grows with their number and
// saturates at the HBM ceiling; each CTA also pays a fixed start-up and finish time, and
// the last CTA of a group pays for the merge -- and picks the split count with the
// shortest simulated step.  It plans for the default schedule: where head-group tiles
// apply (d = 128 with 16- or 32-token pages and Hkv a multiple of 4) a CTA streams one
// split of four kv heads in 16-token tiles, one 16 KB box per K and V.  (The automatic
// schedule also takes head groups -- and, for short rows, their persistent form -- for
// batches of at least 5 (b, kv head) pairs per SM on any cache; both planners already
// give those one split, since one wave of one-head CTAs is full without splitting.)
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <functional>
#include <queue>
#include <vector>

#include "fd.h"

namespace {

constexpr int32_t kMaxSplits = 4096;
constexpr int64_t kMinSplitTokens = 256;
constexpr int kCtasPerSm = 2;             // residency of the partial kernels
constexpr int kHeadGroup = 4;             // kv heads per CTA with head-group tiles

// Model constants, fitted on GB300 to this library's partial kernel: n CTAs streaming
// at once reach BW(n) = kHbmBytesPerUs * (1 - exp(-n / tau)) together, shared equally.
// Contiguous caches: tau = 95 (fitted to 32, 64 and 128 CTAs streaming 2048, 1024 and
// 512 tokens each once their fixed time is taken out; one CTA alone ~72 GB/s; 7.0 TB/s
// is the read ceiling).  Paged caches issue one TMA box
// per page, so one CTA streams slower (~55 GB/s with pages of a tile or more, ~27 GB/s
// with 16-token pages) and tau grows in proportion.
constexpr double kHbmBytesPerUs = 7.0e6;
constexpr double kSatCtasContig = 95.0;
constexpr double kOneCtaContig = 72.5e3;    // bytes per µs
constexpr double kCtaFixedUs = 2.0;         // start-up + epilogue of one CTA
constexpr double kMergeBytesPerUs = 1.0e5;  // merging a group's partials from L2
constexpr double kMisalignedPenalty = 1.04;

// One CTA's streaming rate (bytes per µs) for a page size (0 = contiguous cache).
double one_cta_rate(int page_size, int tile) {
  if (page_size <= 0) return kOneCtaContig;
  if (page_size >= tile) return 55.0e3;
  return std::min(55.0e3, 27.5e3 * page_size / 16.0);
}

double rate_per_cta(size_t n, double tau) {
  return kHbmBytesPerUs * (1.0 - std::exp(-(double)n / tau)) / (double)n;
}

int tile_tokens_bf16(int d) { return 16384 / (d * 2); }

// Simulated duration (µs) of one partial-pass launch.
//   work[i]  bytes CTA i streams (launch order), fixed[i] its fixed time (µs).
double simulate(const std::vector<double>& work, const std::vector<double>& fixed, int slots,
                double tau) {
  // Every running CTA progresses at the same rate, so track the progress P (in bytes;
  // a CTA's fixed time counts as bytes at the one-CTA rate) at which each one finishes.
  std::priority_queue<double, std::vector<double>, std::greater<double>> heap;
  const size_t n = work.size();
  const double fixed_rate = rate_per_cta(1, tau);
  size_t next = 0;
  double t = 0.0, P = 0.0;
  auto push = [&](size_t i) { heap.push(P + work[i] + fixed[i] * fixed_rate); };
  while (next < n && (int)heap.size() < slots) push(next++);
  while (!heap.empty()) {
    const double rate = rate_per_cta(heap.size(), tau);
    const double f = heap.top();
    heap.pop();
    t += (f - P) / rate;
    P = f;
    if (next < n) push(next++);
  }
  return t;
}

// Whether the default schedule runs head-group tiles for these sizes (bf16 assumed).
bool head_groups(int Hkv, int d, int page_size) {
  return d == 128 && (page_size == 16 || page_size == 32) && Hkv % kHeadGroup == 0;
}

// Per-CTA work of one split count: bytes each CTA loads (whole tiles, as the kernels
// do) and its fixed time, in launch order (split fastest, then kv head or head group,
// then row).
double plan_time(int B, int Hq, int Hkv, int d, int64_t L_cap, const int32_t* lens, int S,
                 int slots, int page_size) {
  const bool heads = head_groups(Hkv, d, page_size);
  const int TT = heads ? 16 : tile_tokens_bf16(d);
  const int per_cta = heads ? kHeadGroup : 1;      // kv heads a CTA streams
  const int64_t split_len = (L_cap + S - 1) / S;
  const double tok_bytes = 2.0 * d * 2.0 * per_cta;   // K and V rows, bf16
  const int G = Hq / Hkv;
  std::vector<double> work, fixed;
  work.reserve((size_t)B * Hkv * S);
  fixed.reserve((size_t)B * Hkv * S);
  for (int b = 0; b < B; ++b) {
    const int64_t L = std::min<int64_t>(std::max<int64_t>(lens ? lens[b] : L_cap, 0), L_cap);
    for (int g = 0; g < Hkv; g += per_cta) {
      int last = -1;
      for (int i = 0; i < S; ++i) {
        const int64_t lo = (int64_t)i * split_len, hi = std::min(lo + split_len, L);
        if (lo < hi) {
          const int64_t t0 = lo / TT * TT, t1 = (hi + TT - 1) / TT * TT;
          work.push_back((double)(t1 - t0) * tok_bytes);
          fixed.push_back(kCtaFixedUs);
          last = (int)work.size() - 1;
        } else {
          work.push_back(0.0);
          fixed.push_back(0.1 * kCtaFixedUs);       // an empty split exits at once
        }
      }
      // The group's merge reads G rows of S partials (d + 1 floats each).
      const double merge_us = (double)per_cta * G * S * (d + 1) * 4.0 / kMergeBytesPerUs;
      if (last >= 0) fixed[last] += merge_us;
    }
  }
  // Head-group tiles are one 16 KB box per K and V, like a contiguous cache's.
  const double tau =
      heads ? kSatCtasContig : kSatCtasContig * kOneCtaContig / one_cta_rate(page_size, TT);
  return simulate(work, fixed, slots, tau);
}

}  // namespace

extern "C" {

int32_t fd_num_splits_heuristic(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int64_t L_cap,
                                int32_t num_sms) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || L_cap <= 0 || num_sms <= 0) return 1;
  const int64_t units = (int64_t)B * Hkv;                   // (b, kv head) pairs
  const int64_t slots = (int64_t)kCtasPerSm * num_sms;      // resident CTAs: one wave
  int64_t S_max = slots / units;
  S_max = std::min<int64_t>(S_max, (L_cap + kMinSplitTokens - 1) / kMinSplitTokens);
  S_max = std::min<int64_t>(S_max, kMaxSplits);
  if (S_max <= 1) return 1;
  // Prefer a split count whose split_len is a whole number of tiles, if it keeps at least
  // three quarters of the one-wave maximum.
  const int64_t TT = tile_tokens_bf16(d);
  for (int64_t S = S_max; 4 * S >= 3 * S_max; --S) {
    if (((L_cap + S - 1) / S) % TT == 0) return (int32_t)S;
  }
  return (int32_t)S_max;
}

int32_t fd_num_splits_for_lengths(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int64_t L_cap,
                                  const int32_t* seq_lens, int32_t page_size, int32_t num_sms) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || L_cap <= 0 || num_sms <= 0 || !seq_lens ||
      Hq % Hkv != 0)
    return 1;
  int64_t L_max = 0;
  for (int b = 0; b < B; ++b) L_max = std::max<int64_t>(L_max, std::min<int64_t>(seq_lens[b], L_cap));
  if (L_max <= 0) return 1;
  const int slots = kCtasPerSm * num_sms;
  // Candidates: every count up to 64, then coarser steps; none with splits shorter than
  // kMinSplitTokens of the capacity.
  std::vector<int> cand;
  for (int S = 1; S <= 64; ++S) cand.push_back(S);
  for (int S = 72; S <= 256; S += 8) cand.push_back(S);
  for (int S = 288; S <= 1024; S += 32) cand.push_back(S);
  const int64_t S_cap = std::max<int64_t>(1, (L_cap + kMinSplitTokens - 1) / kMinSplitTokens);
  const int TT = head_groups(Hkv, d, page_size) ? 16 : tile_tokens_bf16(d);
  int best_S = 1;
  double best_t = plan_time(B, Hq, Hkv, d, L_cap, seq_lens, 1, slots, page_size);
  if (L_cap % TT != 0) best_t *= kMisalignedPenalty;
  for (int S : cand) {
    if (S == 1 || S > S_cap || S > kMaxSplits) continue;
    double t = plan_time(B, Hq, Hkv, d, L_cap, seq_lens, S, slots, page_size);
    // A split that ends mid-tile makes two CTAs load its boundary tile and breaks the
    // tiles' alignment; measured on the 128K workload it costs ~4% beyond the extra
    // bytes the model already counts (S = 38: 83.3 us against 79.9 us at S = 32).
    if (((L_cap + S - 1) / S) % TT != 0) t *= kMisalignedPenalty;
    if (t < best_t * 0.995) {                 // a smaller count wins near-ties
      best_t = t;
      best_S = S;
    }
  }
  return best_S;
}

}  // extern "C"
