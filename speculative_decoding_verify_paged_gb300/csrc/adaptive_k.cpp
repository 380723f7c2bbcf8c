// Adaptive draft length, host side ("Speculative decoding principles and a
// vLLM production setup", sec. 4.3): per sequence, a window of the last
// acceptance rates alpha = a / max(K, 1); with enough of them, their mean moves
// K by one step up or down within [k_min, k_max].
//
// The state is one caller-owned block: a header with the parameters, one
// record per sequence (K, rates held, next write slot) and the rings of rates.
// The mean is summed oldest first in double, so two implementations that add
// in that order agree bit for bit.
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstring>

#include "spec_verify.h"

namespace {

constexpr uint64_t kMagic = 0x4b5f5041445f5653ull;  // identifies an initialised state
constexpr int32_t kMaxK = 63;                       // K + 1 query rows <= 64

struct Header {
  uint64_t magic;
  int32_t batch;
  int32_t reserved;
  sv_adaptive_k_params p;
};

struct SeqRec {
  int32_t k;      // K for the next step
  int32_t count;  // rates held, <= window
  int32_t head;   // ring slot of the next rate
  int32_t reserved;
};

constexpr size_t kHeaderBytes = (sizeof(Header) + 63) / 64 * 64;

size_t state_bytes(int64_t batch, int64_t window) {
  if (batch < 0 || window < 1) return 0;
  const int64_t bytes = (int64_t)kHeaderBytes + batch * (int64_t)sizeof(SeqRec) + batch * window * 8;
  if (bytes > ((int64_t)1 << 40)) return 0;
  return (size_t)bytes;
}

SeqRec *seqs(void *state) { return reinterpret_cast<SeqRec *>(static_cast<char *>(state) + kHeaderBytes); }
const SeqRec *seqs(const void *state) {
  return reinterpret_cast<const SeqRec *>(static_cast<const char *>(state) + kHeaderBytes);
}
double *rates(void *state, int32_t batch) {
  return reinterpret_cast<double *>(reinterpret_cast<char *>(seqs(state)) + (size_t)batch * sizeof(SeqRec));
}

bool params_ok(const sv_adaptive_k_params &p) {
  return p.k_min >= 0 && p.k_min <= p.k_init && p.k_init <= p.k_max && p.k_max <= kMaxK && p.window >= 1 &&
         p.min_samples >= 1 && std::isfinite(p.up_threshold) && std::isfinite(p.down_threshold);
}

const Header *header_of(const void *state) {
  if (state == nullptr || (reinterpret_cast<uintptr_t>(state) & 7u) != 0) return nullptr;
  const Header *h = static_cast<const Header *>(state);
  return h->magic == kMagic ? h : nullptr;
}

void reset_seq(SeqRec &s, const sv_adaptive_k_params &p) {
  s.k = p.k_init;
  s.count = 0;
  s.head = 0;
  s.reserved = 0;
}

}  // namespace

extern "C" {

size_t sv_adaptive_k_state_bytes(int32_t batch, int32_t window) { return state_bytes(batch, window); }

sv_status sv_adaptive_k_init(void *state, size_t bytes, int32_t batch, const sv_adaptive_k_params *params) {
  if (state == nullptr || (reinterpret_cast<uintptr_t>(state) & 7u) != 0 || params == nullptr)
    return SV_ERR_INVALID_ARG;
  if (!params_ok(*params)) return SV_ERR_INVALID_ARG;
  const size_t need = state_bytes(batch, params->window);
  if (need == 0 || bytes < need) return SV_ERR_INVALID_ARG;
  Header h;
  std::memset(&h, 0, sizeof h);
  h.magic = kMagic;
  h.batch = batch;
  h.p = *params;
  std::memcpy(state, &h, sizeof h);
  SeqRec *s = seqs(state);
  for (int32_t b = 0; b < batch; ++b) reset_seq(s[b], *params);
  std::memset(rates(state, batch), 0, (size_t)batch * (size_t)params->window * sizeof(double));
  return SV_OK;
}

sv_status sv_adaptive_k_update(void *state, const int32_t *accepted, const int32_t *drafted, int32_t *k_next) {
  const Header *h = header_of(state);
  if (h == nullptr) return SV_ERR_INVALID_ARG;
  const int32_t B = h->batch;
  const sv_adaptive_k_params &p = h->p;
  if (B > 0 && (accepted == nullptr || drafted == nullptr)) return SV_ERR_INVALID_ARG;
  for (int32_t b = 0; b < B; ++b)  // all or nothing
    if (drafted[b] < 0 || accepted[b] < 0 || accepted[b] > drafted[b]) return SV_ERR_INVALID_ARG;
  SeqRec *s = seqs(state);
  double *ring_all = rates(state, B);
  const size_t W = (size_t)p.window;
  // record the step's rates
  for (int32_t b = 0; b < B; ++b) {
    SeqRec &r = s[b];
    const int32_t d = drafted[b] > 1 ? drafted[b] : 1;
    ring_all[(size_t)b * W + r.head] = (double)accepted[b] / (double)d;
    r.head = r.head + 1 == p.window ? 0 : r.head + 1;
    if (r.count < p.window) ++r.count;
  }
  // the means, oldest rate first; sequences whose rings line up (the usual case:
  // the same number of steps since their last reset) are summed eight at a time
  // with independent accumulators, each in the same order as alone
  auto apply = [&](SeqRec &r, double sum) {
    const double mean = sum / (double)r.count;
    if (mean > p.up_threshold) r.k = r.k + 1 < p.k_max ? r.k + 1 : p.k_max;
    else if (mean < p.down_threshold) r.k = r.k - 1 > p.k_min ? r.k - 1 : p.k_min;
  };
  constexpr int kLanes = 8;
  int32_t b = 0;
  while (b < B) {
    const SeqRec &r0 = s[b];
    bool group = b + kLanes <= B;
    for (int j = 1; group && j < kLanes; ++j) group = s[b + j].head == r0.head && s[b + j].count == r0.count;
    if (r0.count >= p.min_samples && group) {
      double acc[kLanes] = {0, 0, 0, 0, 0, 0, 0, 0};
      const double *base = ring_all + (size_t)b * W;
      int32_t i = r0.head - r0.count;
      if (i < 0) i += p.window;
      for (int32_t n = 0; n < r0.count; ++n) {
        for (int j = 0; j < kLanes; ++j) acc[j] += base[(size_t)j * W + i];
        i = i + 1 == p.window ? 0 : i + 1;
      }
      for (int j = 0; j < kLanes; ++j) apply(s[b + j], acc[j]);
      b += kLanes;
      continue;
    }
    const int32_t end = group ? b + kLanes : b + 1;
    for (; b < end; ++b) {
      SeqRec &r = s[b];
      if (r.count < p.min_samples) continue;
      const double *ring = ring_all + (size_t)b * W;
      int32_t i = r.head - r.count;
      if (i < 0) i += p.window;
      double sum = 0.0;
      for (int32_t n = 0; n < r.count; ++n) {
        sum += ring[i];
        i = i + 1 == p.window ? 0 : i + 1;
      }
      apply(r, sum);
    }
  }
  if (k_next != nullptr)
    for (int32_t q = 0; q < B; ++q) k_next[q] = s[q].k;
  return SV_OK;
}

sv_status sv_adaptive_k_reset(void *state, int32_t seq) {
  const Header *h = header_of(state);
  if (h == nullptr || seq < 0 || seq >= h->batch) return SV_ERR_INVALID_ARG;
  reset_seq(seqs(state)[seq], h->p);
  return SV_OK;
}

sv_status sv_adaptive_k_current(const void *state, int32_t *k) {
  const Header *h = header_of(state);
  if (h == nullptr || (h->batch > 0 && k == nullptr)) return SV_ERR_INVALID_ARG;
  const SeqRec *s = seqs(state);
  for (int32_t b = 0; b < h->batch; ++b) k[b] = s[b].k;
  return SV_OK;
}

}  // extern "C"
