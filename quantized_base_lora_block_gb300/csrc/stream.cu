// Layer streaming of a frozen base: pinned host memory -> a fixed pool of
// device slots, copied one layer ahead on a dedicated copy stream, ordered
// against the compute stream with events.
//
// Each slot carries the layer id it holds and a state: empty, pending (copied
// or resident and announced by prefetch, not yet acquired), acquired, or
// released (consumed, may be refilled).  acquire() checks the id, so a slot
// that was refilled with another layer is never read as the old one (a stale
// buffer is an error, not a silent wrong answer).  prefetch() only refills
// empty or released slots, least recently used first; it never evicts a
// pending layer, and fails with QLORA_ERR_STATE when no slot is free.  A layer
// that is still resident is not copied again (the backward pass starts on the
// layers the forward pass ended with).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/qlora.h"
#include "kernels.h"

namespace qlora {

struct StreamPool {
  int slots = 0;
  size_t slot_bytes = 0;
  uint8_t* dev = nullptr;
  cudaStream_t copy = nullptr;
  std::vector<cudaEvent_t> ready;
  // one event per release since the slot was last filled: a slot acquired on
  // several unordered streams is refilled only after every one of them
  std::vector<std::vector<cudaEvent_t>> released;
  std::vector<cudaEvent_t> spare;  // recycled release events
  std::vector<int> layer;     // layer held by the slot, -1 = none
  std::vector<int> acquired;  // compute work holding the slot not yet released
  std::vector<int> pending;   // announced by prefetch, not yet acquired
  std::vector<uint64_t> last_use;
  uint64_t clock = 0;
  std::mutex mu;
};

}  // namespace qlora

using namespace qlora;

extern "C" {

int32_t qlora_stream_create(int32_t slots, size_t slot_bytes, void** handle) {
  if (!handle || slots < 1 || slots > 64 || slot_bytes == 0) return QLORA_ERR_INVALID;
  *handle = nullptr;
  StreamPool* p = new StreamPool();
  p->slots = slots;
  p->slot_bytes = (slot_bytes + 255) & ~size_t(255);
  if (cudaMalloc(&p->dev, p->slot_bytes * slots) != cudaSuccess) {
    delete p;
    return QLORA_ERR_CUDA;
  }
  if (cudaStreamCreateWithFlags(&p->copy, cudaStreamNonBlocking) != cudaSuccess) {
    cudaFree(p->dev);
    delete p;
    return QLORA_ERR_CUDA;
  }
  p->ready.resize(slots);
  p->released.resize(slots);
  for (int i = 0; i < slots; ++i) cudaEventCreateWithFlags(&p->ready[i], cudaEventDisableTiming);
  p->layer.assign(slots, -1);
  p->acquired.assign(slots, 0);
  p->pending.assign(slots, 0);
  p->last_use.assign(slots, 0);
  *handle = p;
  return QLORA_OK;
}

int32_t qlora_stream_prefetch(void* handle, int32_t layer, const void* host_src, size_t bytes) {
  StreamPool* p = static_cast<StreamPool*>(handle);
  if (!p || !host_src || layer < 0) return QLORA_ERR_INVALID;
  if (bytes == 0 || bytes > p->slot_bytes) return QLORA_ERR_INVALID;
  std::lock_guard<std::mutex> g(p->mu);
  for (int i = 0; i < p->slots; ++i)
    if (p->layer[i] == layer) {  // already resident
      p->pending[i] = 1;
      p->last_use[i] = ++p->clock;
      return QLORA_OK;
    }
  int victim = -1;
  for (int i = 0; i < p->slots; ++i) {
    if (p->acquired[i] || p->pending[i]) continue;
    if (victim < 0 || p->last_use[i] < p->last_use[victim]) victim = i;
  }
  if (victim < 0) return QLORA_ERR_STATE;  // every slot is in use or pending
  // the refill waits for every use of the slot released since its last fill
  for (cudaEvent_t e : p->released[victim])
    if (cudaStreamWaitEvent(p->copy, e, 0) != cudaSuccess) return QLORA_ERR_CUDA;
  // the copy stream now holds the waits: the events may be recorded again
  for (cudaEvent_t e : p->released[victim]) p->spare.push_back(e);
  p->released[victim].clear();
  p->layer[victim] = -1;
  if (cudaMemcpyAsync(p->dev + (size_t)victim * p->slot_bytes, host_src, bytes, cudaMemcpyHostToDevice, p->copy) !=
      cudaSuccess)
    return QLORA_ERR_CUDA;
  if (cudaEventRecord(p->ready[victim], p->copy) != cudaSuccess) return QLORA_ERR_CUDA;
  p->layer[victim] = layer;
  p->pending[victim] = 1;
  p->last_use[victim] = ++p->clock;
  return QLORA_OK;
}

int32_t qlora_stream_acquire(void* handle, int32_t layer, void* compute_stream, void** dev_ptr) {
  StreamPool* p = static_cast<StreamPool*>(handle);
  if (!p || !dev_ptr) return QLORA_ERR_INVALID;
  std::lock_guard<std::mutex> g(p->mu);
  for (int i = 0; i < p->slots; ++i) {
    if (p->layer[i] != layer) continue;
    if (cudaStreamWaitEvent(static_cast<cudaStream_t>(compute_stream), p->ready[i], 0) != cudaSuccess)
      return QLORA_ERR_CUDA;
    p->acquired[i] += 1;
    p->pending[i] = 0;
    p->last_use[i] = ++p->clock;
    *dev_ptr = p->dev + (size_t)i * p->slot_bytes;
    return QLORA_OK;
  }
  *dev_ptr = nullptr;
  return QLORA_ERR_STATE;
}

int32_t qlora_stream_release(void* handle, int32_t layer, void* compute_stream) {
  StreamPool* p = static_cast<StreamPool*>(handle);
  if (!p) return QLORA_ERR_INVALID;
  std::lock_guard<std::mutex> g(p->mu);
  for (int i = 0; i < p->slots; ++i) {
    if (p->layer[i] != layer || p->acquired[i] == 0) continue;
    cudaEvent_t e = nullptr;
    if (!p->spare.empty()) {
      e = p->spare.back();
      p->spare.pop_back();
    } else if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      return QLORA_ERR_CUDA;
    }
    if (cudaEventRecord(e, static_cast<cudaStream_t>(compute_stream)) != cudaSuccess) {
      p->spare.push_back(e);
      return QLORA_ERR_CUDA;
    }
    p->released[i].push_back(e);
    p->acquired[i] -= 1;
    return QLORA_OK;
  }
  return QLORA_ERR_STATE;
}

int32_t qlora_stream_destroy(void* handle) {
  StreamPool* p = static_cast<StreamPool*>(handle);
  if (!p) return QLORA_ERR_INVALID;
  cudaStreamSynchronize(p->copy);
  for (int i = 0; i < p->slots; ++i) {
    for (cudaEvent_t e : p->released[i]) {
      cudaEventSynchronize(e);
      cudaEventDestroy(e);
    }
    cudaEventDestroy(p->ready[i]);
  }
  for (cudaEvent_t e : p->spare) cudaEventDestroy(e);
  cudaStreamDestroy(p->copy);
  cudaFree(p->dev);
  delete p;
  return QLORA_OK;
}

}  // extern "C"
