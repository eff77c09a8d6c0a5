// Host-side checks of the slot-id contract that the kernels do not check themselves: the slot ids of one
// call are distinct, and the slots a copy or a snapshot writes are not the slots it reads from the same
// pool.  "SGLang and Miles: day-0 support for Kimi K3", three state movements on the forward stream: a
// snapshot's target slot is never the slot it is taken from, and every request owns its slot.
//
// Off by default (the calls stay asynchronous and capturable).  With the checks on (kda_set_debug_checks(1),
// or KDA_DEBUG_CHECKS=1 in the environment at the first call), an entry point that takes slot ids first
// copies them to the host on its stream, waits for that copy, and returns KDA_ERR_INVALID_ARG without
// enqueuing anything when the contract is broken.
#include <stdint.h>
#include <stdlib.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include "../../include/kda.h"
#include "debug_checks.h"

namespace {

std::atomic<int> g_debug{-1};  // -1: not yet read from the environment

bool sorted_has_duplicate(std::vector<int32_t>& v) {
  std::sort(v.begin(), v.end());
  return std::adjacent_find(v.begin(), v.end()) != v.end();
}

}  // namespace

extern "C" {

kda_status kda_check_slot_ids(const int32_t* ids, int32_t n, const int32_t* other_ids, int32_t n_other) {
  if (n < 0 || n_other < 0 || (n > 0 && !ids) || (n_other > 0 && !other_ids)) return KDA_ERR_INVALID_ARG;
  std::vector<int32_t> a(ids, ids + n);
  if (sorted_has_duplicate(a)) return KDA_ERR_INVALID_ARG;
  if (n_other > 0) {
    std::vector<int32_t> b(other_ids, other_ids + n_other);
    std::sort(b.begin(), b.end());
    std::vector<int32_t> both;
    std::set_intersection(a.begin(), a.end(), b.begin(), b.end(), std::back_inserter(both));
    if (!both.empty()) return KDA_ERR_INVALID_ARG;
  }
  return KDA_OK;
}

void kda_set_debug_checks(int on) { g_debug.store(on ? 1 : 0); }

int kda_debug_checks(void) {
  int v = g_debug.load();
  if (v < 0) {
    const char* e = getenv("KDA_DEBUG_CHECKS");
    v = (e && e[0] && e[0] != '0') ? 1 : 0;
    int expected = -1;
    g_debug.compare_exchange_strong(expected, v);
    v = g_debug.load();
  }
  return v;
}

}  // extern "C"

namespace kda {

namespace {
// Copies n device ids to `out` on the stream and waits for them.
bool fetch_ids(const int32_t* dev_ids, int32_t n, std::vector<int32_t>& out, cudaStream_t s) {
  out.resize(n > 0 ? n : 0);
  if (n <= 0) return true;
  if (cudaMemcpyAsync(out.data(), dev_ids, (size_t)n * sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return false;
  return cudaStreamSynchronize(s) == cudaSuccess;
}
}  // namespace

kda_status debug_check_slots(const int32_t* dev_ids, int32_t n, const int32_t* dev_other, int32_t n_other,
                             cudaStream_t s) {
  if (!kda_debug_checks()) return KDA_OK;
  std::vector<int32_t> a, b;
  if (!fetch_ids(dev_ids, n, a, s)) return KDA_ERR_CUDA;
  if (dev_other && !fetch_ids(dev_other, n_other, b, s)) return KDA_ERR_CUDA;
  return kda_check_slot_ids(a.data(), n, dev_other ? b.data() : nullptr, dev_other ? n_other : 0);
}

}  // namespace kda
