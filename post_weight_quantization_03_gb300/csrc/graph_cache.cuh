// A few captured CUDA graphs of one enqueue routine, keyed by the routine's arguments.
//
// The factorization's panel loop and the blocked sweep are long chains of dependent launches
// on several streams; replaying a chain as one captured graph removes most of the launch
// latency between its kernels.  The graph is captured on (and launched on) one of the
// library's own streams, so the caller's stream can be any stream, the legacy default one
// included; the caller joins it to that stream with events on both sides.
#pragma once

#include <algorithm>
#include <vector>

#include "common.cuh"

namespace gptq {

unsigned long long launches_so_far();

struct GraphCache {
  struct Entry {
    cudaGraphExec_t exec = nullptr;
    std::vector<uint64_t> key;
    unsigned kernels = 0;        // kernel launches the graph holds
    unsigned long long used = 0;
  };
  static constexpr int kEntries = 8;
  Entry entries[kEntries];
  unsigned long long tick = 0;

  // Launches enqueue(origin) as a graph on `origin`, capturing it first when no entry has
  // this key.  Returns false (nothing launched, errors cleared) when capture or
  // instantiation fails; the caller then enqueues directly.  `status` receives the status of
  // a failed enqueue during capture.
  template <class F>
  bool run(const std::vector<uint64_t> &key, cudaStream_t origin, F &&enqueue,
           gptq_status *status) {
    Entry *hit = nullptr, *lru = &entries[0];
    for (Entry &e : entries) {
      if (e.exec && e.key == key) hit = &e;
      if (e.used < lru->used) lru = &e;
    }
    if (!hit) {
      cudaGraph_t g = nullptr;
      cudaGraphExec_t exec = nullptr;
      const unsigned long long n0 = launches_so_far();
      gptq_status st = GPTQ_ERR_CUDA;
      if (cudaStreamBeginCapture(origin, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
        st = enqueue(origin);
        if (cudaStreamEndCapture(origin, &g) != cudaSuccess) st = GPTQ_ERR_CUDA;
      }
      // kernel nodes keep the priority of the stream they were captured on (critical chain
      // over side work); without this flag the whole graph runs at the launch stream's
      if (st != GPTQ_OK || !g ||
          cudaGraphInstantiateWithFlags(&exec, g, cudaGraphInstantiateFlagUseNodePriority) !=
              cudaSuccess) {
        (void)cudaGetLastError();
        if (g) cudaGraphDestroy(g);
        if (status) *status = st;
        return false;
      }
      cudaGraphDestroy(g);
      hit = lru;
      if (hit->exec) cudaGraphExecDestroy(hit->exec);
      hit->exec = exec;
      hit->key = key;
      hit->kernels = (unsigned)(launches_so_far() - n0);  // counted while capturing
    } else {
      count_launch(hit->kernels);
    }
    hit->used = ++tick;
    if (cudaGraphLaunch(hit->exec, origin) != cudaSuccess) {
      (void)cudaGetLastError();
      if (status) *status = GPTQ_ERR_CUDA;
      return false;
    }
    return true;
  }
};

// True when `s` is being captured by the caller (then everything is launched directly, and
// the caller's capture records it).
inline bool caller_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    (void)cudaGetLastError();
    return true;
  }
  return cap != cudaStreamCaptureStatusNone;
}

}  // namespace gptq
