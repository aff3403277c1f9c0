// Pipelined expert forward on host-resident batches: the host -> device copy
// of step i + 1 and the device -> host copy of step i - 1 overlap the
// forward of step i.
//
// Three streams: copy-in, compute, copy-out.  Slot s = i % depth holds step
// i's device copies of x and the logits and its output.  Events order each
// slot's reuse: the copy-in of step i waits until the forward of step
// i - depth has finished reading the slot, and the forward of step i waits
// for its own copy-in and for the copy-out of step i - depth from the slot's
// output buffer.  The forwards run in submission order on the compute
// stream, so they share one workspace.  Nothing is allocated: the caller
// passes one device buffer for the slots and the workspace; streams and
// events are created once, at moe_pipeline_create.
#include <new>

#include "common.cuh"

struct moe_pipeline {
  int T, E, k, d, d_ff, depth, device;
  uint16_t* x[MOE_PIPELINE_MAX_DEPTH];
  float* logits[MOE_PIPELINE_MAX_DEPTH];
  uint16_t* out[MOE_PIPELINE_MAX_DEPTH];
  void* ws;
  size_t ws_bytes;
  cudaStream_t in, comp, outs;
  cudaEvent_t ev_in[MOE_PIPELINE_MAX_DEPTH], ev_comp[MOE_PIPELINE_MAX_DEPTH], ev_out[MOE_PIPELINE_MAX_DEPTH];
  bool used[MOE_PIPELINE_MAX_DEPTH];
  unsigned long long steps;
};

namespace {

inline size_t up1024(size_t x) { return (x + 1023) & ~size_t(1023); }

struct SlotSizes {
  size_t x, logits, out, slot;
};

SlotSizes slot_sizes(int T, int E, int d) {
  SlotSizes s;
  s.x = up1024((size_t)T * d * 2);
  s.logits = up1024((size_t)T * E * 4);
  s.out = up1024((size_t)T * d * 2);
  s.slot = s.x + s.logits + s.out;
  return s;
}

bool ok_pipe_shape(int T, int depth) { return T >= 1 && depth >= 1 && depth <= MOE_PIPELINE_MAX_DEPTH; }

void release(moe_pipeline* p) {
  for (int s = 0; s < MOE_PIPELINE_MAX_DEPTH; ++s) {
    if (p->ev_in[s]) cudaEventDestroy(p->ev_in[s]);
    if (p->ev_comp[s]) cudaEventDestroy(p->ev_comp[s]);
    if (p->ev_out[s]) cudaEventDestroy(p->ev_out[s]);
  }
  if (p->in) cudaStreamDestroy(p->in);
  if (p->comp) cudaStreamDestroy(p->comp);
  if (p->outs) cudaStreamDestroy(p->outs);
  delete p;
}

}  // namespace

extern "C" {

size_t moe_pipeline_device_bytes(int T, int E, int k, int d, int d_ff, int depth) {
  if (!ok_pipe_shape(T, depth)) return 0;
  const size_t ws = moe_expert_forward_workspace_bytes(T, E, k, d, d_ff);
  if (ws == 0) return 0;
  return (size_t)depth * slot_sizes(T, E, d).slot + up1024(ws);
}

int moe_pipeline_create(int T, int E, int k, int d, int d_ff, int depth, void* device_buffer, size_t bytes,
                        moe_pipeline** out) {
  if (!out || !device_buffer || (reinterpret_cast<uintptr_t>(device_buffer) & 1023u) != 0) return MOE_ERR_POINTER;
  *out = nullptr;
  const size_t need = moe_pipeline_device_bytes(T, E, k, d, d_ff, depth);
  if (need == 0) return MOE_ERR_SHAPE;
  if (bytes < need) return MOE_ERR_WORKSPACE;
  moe_pipeline* p = new (std::nothrow) moe_pipeline();
  if (!p) return MOE_ERR_CUDA;
  p->T = T; p->E = E; p->k = k; p->d = d; p->d_ff = d_ff; p->depth = depth;
  if (cudaGetDevice(&p->device) != cudaSuccess) { release(p); return MOE_ERR_CUDA; }
  const SlotSizes ss = slot_sizes(T, E, d);
  uint8_t* b = static_cast<uint8_t*>(device_buffer);
  for (int s = 0; s < depth; ++s) {
    uint8_t* base = b + (size_t)s * ss.slot;
    p->x[s] = reinterpret_cast<uint16_t*>(base);
    p->logits[s] = reinterpret_cast<float*>(base + ss.x);
    p->out[s] = reinterpret_cast<uint16_t*>(base + ss.x + ss.logits);
  }
  p->ws = b + (size_t)depth * ss.slot;
  p->ws_bytes = moe_expert_forward_workspace_bytes(T, E, k, d, d_ff);
  bool ok = cudaStreamCreateWithFlags(&p->in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->comp, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->outs, cudaStreamNonBlocking) == cudaSuccess;
  for (int s = 0; ok && s < depth; ++s)
    ok = cudaEventCreateWithFlags(&p->ev_in[s], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->ev_comp[s], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->ev_out[s], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    release(p);
    return MOE_ERR_CUDA;
  }
  *out = p;
  return MOE_OK;
}

int moe_pipeline_submit(moe_pipeline* p, const uint16_t* host_x, const float* host_logits, uint16_t* host_out,
                        const uint8_t* w1_codes, const uint8_t* w1_sf, const float* w1_g, const uint8_t* w2_codes,
                        const uint8_t* w2_sf, const float* w2_g, int* status) {
  if (!p || !host_x || !host_logits || !host_out) return MOE_ERR_POINTER;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev != p->device) return MOE_ERR_DEVICE;
  const int s = (int)(p->steps % (unsigned long long)p->depth);
  const int T = p->T, d = p->d, E = p->E;
  if (p->used[s] && cudaStreamWaitEvent(p->in, p->ev_comp[s], 0) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(p->x[s], host_x, (size_t)T * d * 2, cudaMemcpyHostToDevice, p->in) != cudaSuccess ||
      cudaMemcpyAsync(p->logits[s], host_logits, (size_t)T * E * 4, cudaMemcpyHostToDevice, p->in) != cudaSuccess ||
      cudaEventRecord(p->ev_in[s], p->in) != cudaSuccess || cudaStreamWaitEvent(p->comp, p->ev_in[s], 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (p->used[s] && cudaStreamWaitEvent(p->comp, p->ev_out[s], 0) != cudaSuccess) return MOE_ERR_CUDA;
  const int rc = moe_expert_forward(p->x[s], p->logits[s], T, E, p->k, d, p->d_ff, w1_codes, w1_sf, w1_g, w2_codes,
                                    w2_sf, w2_g, p->out[s], p->ws, p->ws_bytes, status, p->comp);
  if (rc != MOE_OK) return rc;
  if (cudaEventRecord(p->ev_comp[s], p->comp) != cudaSuccess ||
      cudaStreamWaitEvent(p->outs, p->ev_comp[s], 0) != cudaSuccess ||
      cudaMemcpyAsync(host_out, p->out[s], (size_t)T * d * 2, cudaMemcpyDeviceToHost, p->outs) != cudaSuccess ||
      cudaEventRecord(p->ev_out[s], p->outs) != cudaSuccess)
    return MOE_ERR_CUDA;
  p->used[s] = true;
  ++p->steps;
  return MOE_OK;
}

int moe_pipeline_synchronize(moe_pipeline* p) {
  if (!p) return MOE_ERR_POINTER;
  if (cudaStreamSynchronize(p->in) != cudaSuccess || cudaStreamSynchronize(p->comp) != cudaSuccess ||
      cudaStreamSynchronize(p->outs) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_pipeline_destroy(moe_pipeline* p) {
  if (!p) return MOE_OK;
  const int rc = moe_pipeline_synchronize(p);
  release(p);
  return rc;
}

}  // extern "C"
