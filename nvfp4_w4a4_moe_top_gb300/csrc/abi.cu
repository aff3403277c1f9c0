// C ABI of libmoe_nvfp4.so (declared in include/moe_nvfp4.h): argument
// validation on the host, TMA tensor-map encoding, workspace layout and the
// launch sequence of each entry point.  No allocation, no synchronisation.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace {

using moe::kRouteChunk;

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool ok_ptr(const void* p) { return p != nullptr && al16(p); }
inline bool ok_opt(const void* p) { return p == nullptr || al16(p); }
inline size_t up1024(size_t x) { return (x + 1023) & ~size_t(1023); }

int64_t m_cap_of(int64_t T, int64_t E, int64_t k) {
  const int64_t routed = T * k;
  const int64_t nonempty = E < routed ? E : routed;
  const int64_t m = routed + 127 * nonempty;
  return (m + 127) / 128 * 128;
}

size_t sf_bytes_of(int64_t rows, int K) { return (size_t)((rows + 127) / 128) * (size_t)(K / 64) * 512; }

bool ok_model_shape(int T, int E, int k, int d, int d_ff) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return false;
  if (d < 128 || d > 4096 || d % 128 != 0) return false;
  if (d_ff < 128 || d_ff > 4096 || d_ff % 128 != 0) return false;
  const int64_t mc = m_cap_of(T, E, k);
  if (mc >= (int64_t(1) << 31) || (int64_t)T * k * d >= (int64_t(1) << 40)) return false;
  return true;
}

// ---- device checks and driver entry point for tensor maps ----
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
int g_dev_ok[64];  // 0 unknown, 1 ok, -1 not sm_103

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MOE_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_dev_ok[dev] == 0) {
    int maj = 0, min = 0;
    if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    g_dev_ok[dev] = (maj == 10 && min == 3) ? 1 : -1;
  }
  if (g_dev_ok[dev] < 0) return MOE_ERR_DEVICE;
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return MOE_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return MOE_OK;
}

// A second stream per host thread and device, with its fork and join
// events, on which the backward copies the permuted x rows while the GEMMs
// before the one that reads them run (created on first use, kept for the
// thread's life).  Returns false where it cannot be created; the caller then
// stays on its own stream.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool tried = false;
};
bool side_stream(SideStream*& out) {
  thread_local SideStream side[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  SideStream& ss = side[dev];
  if (!ss.tried) {
    ss.tried = true;
    if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess) {
      (void)cudaGetLastError();
      ss.s = nullptr;
    }
  }
  out = &ss;
  return ss.s != nullptr;
}

// 2-D byte tensor of `rows` rows of `row_bytes` bytes, read in boxes of
// 128 rows x 128 bytes with the 128-byte swizzle (the K-major operand layout
// the tensor cores read).
int encode_operand(CUtensorMap* map, const void* base, int64_t rows, int row_bytes) {
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {128u, 128u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// 2-D BF16 tensor of `rows` x `cols` (row-major), read in boxes of
// box_rows rows x 64 columns (128 bytes) with the 128-byte swizzle.
int encode_bf16(CUtensorMap* map, const void* base, int64_t rows, int cols, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// Token-ordered codes (`rows` rows of `row_bytes`) read by tile::gather4:
// boxes of one row x 128 bytes, 128-byte swizzle.
int encode_gather_rows(CUtensorMap* map, const void* base, int64_t rows, int row_bytes) {
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {128u, 1u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// FP32 output [rows][cols] written by TMA stores of 32 x 32 boxes (128-byte
// rows, 128-byte swizzle).
int encode_f32_out(CUtensorMap* map, void* base, int64_t rows, int cols) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  const cuuint32_t box[2] = {32u, 32u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

int finish() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

struct FwdLayout {
  size_t off[16];
  size_t total;
};

FwdLayout fwd_layout(int T, int E, int k, int d, int d_ff) {
  const int64_t mc = m_cap_of(T, E, k);
  const int64_t C = (T + kRouteChunk - 1) / kRouteChunk;
  const size_t sizes[16] = {
      (size_t)T * k * 4, (size_t)T * k * 4, (size_t)T * k * 4, (size_t)E * 4, (size_t)(E + 1) * 4, (size_t)mc * 4,
      (size_t)T * 4,     (size_t)mc * (d / 2), sf_bytes_of(mc, d), (size_t)mc * 4, (size_t)mc * (d_ff / 2),
      sf_bytes_of(mc, d_ff), (size_t)mc * 4, (size_t)mc * d * 2, (size_t)C * E * 4,
      moe::fc1_workspace_bytes(d_ff)};
  FwdLayout L;
  size_t o = 0;
  for (int i = 0; i < 16; ++i) {
    L.off[i] = o;
    o += up1024(sizes[i]);
  }
  L.total = o;
  return L;
}

struct BwdLayout {
  size_t off[4];  // dy2 bf16 [mc][d], xp bf16 [mc][d], du bf16 [mc][2 d_ff], dxr f32 [mc][d]
  size_t total;
};

BwdLayout bwd_layout(int T, int E, int k, int d, int d_ff) {
  const int64_t mc = m_cap_of(T, E, k);
  const size_t sizes[4] = {(size_t)mc * d * 2, (size_t)mc * d * 2, (size_t)mc * 2 * d_ff * 2, (size_t)mc * d * 4};
  BwdLayout L;
  size_t o = 0;
  for (int i = 0; i < 4; ++i) {
    L.off[i] = o;
    o += up1024(sizes[i]);
  }
  L.total = o;
  return L;
}

// The forward of moe_expert_forward; with save_u / save_h / save_y2 set it
// also keeps the values the backward needs.
int forward_impl(const uint16_t* x, const float* logits, int T, int E, int k, int d, int d_ff,
                 const uint8_t* w1_codes, const uint8_t* w1_sf, const float* w1_g, const uint8_t* w2_codes,
                 const uint8_t* w2_sf, const float* w2_g, uint16_t* out, void* ws, size_t ws_bytes, uint16_t* save_u,
                 uint16_t* save_h, float* save_y2, bool gather, int* status, void* stream,
                 void* const* events = nullptr);

}  // namespace

extern "C" {

int moe_abi_version(void) { return MOE_NVFP4_ABI_VERSION; }

const char* moe_status_string(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_POINTER: return "null or misaligned pointer (16-byte alignment required)";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime or launch error";
    case MOE_ERR_DEVICE: return "device is not compute capability 10.3 (sm_103)";
    default: return "unknown status";
  }
}

int64_t moe_m_cap(int T, int E, int k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  return m_cap_of(T, E, k);
}

size_t nvfp4_sf_bytes(int64_t rows, int K) {
  if (rows < 0 || K < 64 || K % 64 != 0) return 0;
  return sf_bytes_of(rows, K);
}

size_t moe_permute_workspace_bytes(int T, int E) {
  if (T < 0 || E < 1) return 0;
  return up1024((size_t)((T + kRouteChunk - 1) / kRouteChunk) * E * 4);
}

size_t nvfp4_fc1_workspace_bytes(int d_ff) {
  if (d_ff < 128 || d_ff % 128 != 0) return 0;
  return moe::fc1_workspace_bytes(d_ff);
}

size_t moe_expert_forward_workspace_bytes(int T, int E, int k, int d, int d_ff) {
  if (!ok_model_shape(T, E, k, d, d_ff)) return 0;
  return fwd_layout(T, E, k, d, d_ff).total;
}

int moe_expert_forward_workspace_layout(int T, int E, int k, int d, int d_ff, size_t offsets_out[16]) {
  if (!offsets_out) return MOE_ERR_POINTER;
  if (!ok_model_shape(T, E, k, d, d_ff)) return MOE_ERR_SHAPE;
  const FwdLayout L = fwd_layout(T, E, k, d, d_ff);
  for (int i = 0; i < 16; ++i) offsets_out[i] = L.off[i];
  return MOE_OK;
}

int moe_nvfp4_quantize_weights(const uint16_t* W, int E, int N, int K, uint8_t* codes, uint8_t* sf, float* g,
                               int* status, void* stream) {
  if (!ok_ptr(W) || !ok_ptr(codes) || !ok_ptr(sf) || !ok_ptr(g) || !ok_opt(status)) return MOE_ERR_POINTER;
  if (E < 1 || N < 128 || N % 128 != 0 || K < 64 || K > 4096 || K % 64 != 0 || (int64_t)E * N >= (int64_t(1) << 31))
    return MOE_ERR_SHAPE;
  int rc = check_device();
  if (rc != MOE_OK) return rc;
  moe::launch_quantize_rows(W, (int64_t)E * N, K, nullptr, nullptr, 1, (int64_t)E * N, codes, sf, g, status,
                            MOE_STATUS_NONFINITE_WEIGHT, (cudaStream_t)stream);
  return finish();
}

int moe_nvfp4_quantize_weights_per_expert(const uint16_t* W, int E, int N, int K, uint8_t* codes, uint8_t* sf,
                                          float* g, float* amax_e, int* status, void* stream) {
  if (!ok_ptr(W) || !ok_ptr(codes) || !ok_ptr(sf) || !ok_ptr(g) || !ok_ptr(amax_e) || !ok_opt(status))
    return MOE_ERR_POINTER;
  if (E < 1 || N < 128 || N % 128 != 0 || K < 64 || K > 4096 || K % 64 != 0 || (int64_t)E * N >= (int64_t(1) << 31))
    return MOE_ERR_SHAPE;
  int rc = check_device();
  if (rc != MOE_OK) return rc;
  if (moe::launch_quantize_weights_per_expert(W, E, N, K, codes, sf, g, amax_e, status, (cudaStream_t)stream) != 0)
    return MOE_ERR_CUDA;
  return finish();
}

int nvfp4_quantize_rows(const uint16_t* src, int src_rows, int K, const int32_t* row_map, const float* amax,
                        int dst_rows, uint8_t* codes, uint8_t* sf, float* g, int* status, void* stream) {
  if (!ok_ptr(src) || !ok_ptr(codes) || !ok_ptr(sf) || !ok_ptr(g) || !ok_opt(row_map) || !ok_opt(amax) ||
      !ok_opt(status))
    return MOE_ERR_POINTER;
  if (src_rows < 1 || dst_rows < 0 || K < 64 || K > 4096 || K % 64 != 0) return MOE_ERR_SHAPE;
  if (!row_map && dst_rows > src_rows) return MOE_ERR_SHAPE;
  int rc = check_device();
  if (rc != MOE_OK) return rc;
  moe::launch_quantize_rows(src, src_rows, K, row_map, amax, 1, dst_rows, codes, sf, g, status, MOE_STATUS_NONFINITE_X,
                            (cudaStream_t)stream);
  return finish();
}

int moe_permute_amax(const float* logits, const int32_t* ext_ids, const float* ext_w, const uint16_t* x, int T, int E,
                     int k, int d, int32_t* topk_ids, float* topk_w, int32_t* counts, int32_t* offsets,
                     int32_t* row_to_token, int32_t* token_slot_row, float* amax_tok, float* amax_row, void* ws,
                     size_t ws_bytes, int* status, void* stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return MOE_ERR_SHAPE;
  if (x && (d < 64 || d > 8192 || d % 64 != 0)) return MOE_ERR_SHAPE;
  if (m_cap_of(T, E, k) >= (int64_t(1) << 31)) return MOE_ERR_SHAPE;
  if (!ok_opt(logits) || !ok_opt(ext_ids) || !ok_opt(ext_w) || !ok_opt(x) || !ok_ptr(counts) || !ok_ptr(offsets) ||
      !ok_opt(status))
    return MOE_ERR_POINTER;
  if (T > 0 && (!ok_ptr(topk_ids) || !ok_ptr(topk_w) || !ok_ptr(row_to_token) || !ok_ptr(token_slot_row) ||
                !ok_ptr(ws)))
    return MOE_ERR_POINTER;
  if (T > 0 && !logits && (!ext_ids || !ext_w)) return MOE_ERR_POINTER;
  if (x && T > 0 && (!ok_ptr(amax_tok) || !ok_ptr(amax_row))) return MOE_ERR_POINTER;
  if (ws_bytes < moe_permute_workspace_bytes(T, E)) return MOE_ERR_WORKSPACE;
  int rc = check_device();
  if (rc != MOE_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t mc = m_cap_of(T, E, k);
  const int C = (T + kRouteChunk - 1) / kRouteChunk;
  int32_t* hist = static_cast<int32_t*>(ws);
  if (T == 0) {
    if (cudaMemsetAsync(counts, 0, (size_t)E * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(offsets, 0, (size_t)(E + 1) * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
    return finish();
  }
  moe::launch_route(logits, ext_ids, ext_w, T, E, k, topk_ids, topk_w, token_slot_row, hist, status, s);
  moe::launch_scan(hist, C, E, counts, s);
  moe::launch_pad_rows(offsets, counts, E, mc, row_to_token, x ? amax_row : nullptr, nullptr, 64, nullptr, nullptr, s);
  moe::launch_permute_amax(topk_ids, token_slot_row, hist, offsets, T, E, k, x, d, row_to_token,
                           x ? amax_tok : nullptr, x ? amax_row : nullptr, status, s);
  return finish();
}

int nvfp4_grouped_gemm_fc1_swiglu(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_g,
                                  const int32_t* offsets, int E, int64_t M_cap, int d, int d_ff,
                                  const uint8_t* w1_codes, const uint8_t* w1_sf, const float* w1_g, uint8_t* h_codes,
                                  uint8_t* h_sf, float* h_g, float* dbg_u_f32, uint16_t* dbg_h, void* ws,
                                  size_t ws_bytes, int* status, void* stream) {
  if (!ok_ptr(a_codes) || !ok_ptr(a_sf) || !ok_ptr(a_g) || !ok_ptr(offsets) || !ok_ptr(w1_codes) || !ok_ptr(w1_sf) ||
      !ok_ptr(w1_g) || !ok_ptr(h_codes) || !ok_ptr(h_sf) || !ok_ptr(h_g) || !ok_opt(dbg_u_f32) || !ok_opt(dbg_h) ||
      !ok_ptr(ws) || !ok_opt(status))
    return MOE_ERR_POINTER;
  if (E < 1 || E > 1024 || M_cap < 128 || M_cap % 128 != 0 || M_cap >= (int64_t(1) << 31) || d < 128 || d > 4096 ||
      d % 128 != 0 || d_ff < 128 || d_ff > 4096 || d_ff % 128 != 0)
    return MOE_ERR_SHAPE;
  if (ws_bytes < nvfp4_fc1_workspace_bytes(d_ff)) return MOE_ERR_WORKSPACE;
  int rc = check_device();
  if (rc != MOE_OK) return rc;
  moe::Fc1Args a;
  std::memset(&a, 0, sizeof(a));
  if (encode_operand(&a.tmap_a, a_codes, M_cap, d / 2) != MOE_OK) return MOE_ERR_CUDA;
  if (encode_operand(&a.tmap_b, w1_codes, (int64_t)E * 2 * d_ff, d / 2) != MOE_OK) return MOE_ERR_CUDA;
  a.a_sf = a_sf; a.a_g = a_g; a.w_sf = w1_sf; a.w_g = w1_g; a.offsets = offsets;
  a.E = E; a.d = d; a.d_ff = d_ff;
  a.h_codes = h_codes; a.h_sf = h_sf; a.h_g = h_g; a.dbg_u = dbg_u_f32; a.dbg_h = dbg_h;
  a.scratch = static_cast<uint16_t*>(ws);
  a.status = status;
  if (moe::launch_fc1(a, M_cap, (cudaStream_t)stream) != 0) return MOE_ERR_CUDA;
  return finish();
}

int nvfp4_grouped_gemm_fc2_unpermute(const uint8_t* h_codes, const uint8_t* h_sf, const float* h_g,
                                     const int32_t* offsets, int E, int64_t M_cap, int d_ff, int d,
                                     const uint8_t* w2_codes, const uint8_t* w2_sf, const float* w2_g,
                                     const int32_t* row_to_token, const int32_t* token_slot_row, const float* topk_w,
                                     int T, int k, uint16_t* slots, uint16_t* out, float* dbg_y_f32, int* status,
                                     void* stream) {
  if (!ok_ptr(h_codes) || !ok_ptr(h_sf) || !ok_ptr(h_g) || !ok_ptr(offsets) || !ok_ptr(w2_codes) || !ok_ptr(w2_sf) ||
      !ok_ptr(w2_g) || !ok_ptr(row_to_token) || !ok_opt(dbg_y_f32) || !ok_opt(status))
    return MOE_ERR_POINTER;
  if (T > 0 && (!ok_ptr(token_slot_row) || !ok_ptr(topk_w) || !ok_ptr(slots) || !ok_ptr(out))) return MOE_ERR_POINTER;
  if (E < 1 || E > 1024 || M_cap < 128 || M_cap % 128 != 0 || M_cap >= (int64_t(1) << 31) || d < 128 || d > 4096 ||
      d % 128 != 0 || d_ff < 128 || d_ff > 4096 || d_ff % 128 != 0 || T < 0 || k < 1 || k > 32 || k > E)
    return MOE_ERR_SHAPE;
  int rc = check_device();
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  moe::Fc2Args a;
  std::memset(&a, 0, sizeof(a));
  if (encode_operand(&a.tmap_a, h_codes, M_cap, d_ff / 2) != MOE_OK) return MOE_ERR_CUDA;
  if (encode_operand(&a.tmap_b, w2_codes, (int64_t)E * d, d_ff / 2) != MOE_OK) return MOE_ERR_CUDA;
  a.a_sf = h_sf; a.a_g = h_g; a.w_sf = w2_sf; a.w_g = w2_g; a.offsets = offsets;
  a.E = E; a.d_ff = d_ff; a.d = d; a.k = k;
  a.row_to_token = row_to_token; a.token_slot_row = token_slot_row; a.topk_w = topk_w;
  a.dbg_y = dbg_y_f32; a.status = status;
  if (encode_bf16(&a.tmap_out, slots, M_cap, d, 32) != MOE_OK) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  if (moe::launch_fc2(a, M_cap, s) != 0) return MOE_ERR_CUDA;
  moe::launch_unpermute_reduce(slots, token_slot_row, T, k, d, out, s);
  return finish();
}

int moe_expert_forward(const uint16_t* x, const float* logits, int T, int E, int k, int d, int d_ff,
                       const uint8_t* w1_codes, const uint8_t* w1_sf, const float* w1_g, const uint8_t* w2_codes,
                       const uint8_t* w2_sf, const float* w2_g, uint16_t* out, void* ws, size_t ws_bytes, int* status,
                       void* stream) {
  return forward_impl(x, logits, T, E, k, d, d_ff, w1_codes, w1_sf, w1_g, w2_codes, w2_sf, w2_g, out, ws, ws_bytes,
                      nullptr, nullptr, nullptr, false, status, stream);
}

int moe_expert_forward_timed(const uint16_t* x, const float* logits, int T, int E, int k, int d, int d_ff,
                             const uint8_t* w1_codes, const uint8_t* w1_sf, const float* w1_g,
                             const uint8_t* w2_codes, const uint8_t* w2_sf, const float* w2_g, uint16_t* out,
                             void* ws, size_t ws_bytes, int* status, void* stream, void* const* events) {
  if (events == nullptr) return MOE_ERR_POINTER;
  for (int i = 0; i < 8; ++i)
    if (events[i] == nullptr) return MOE_ERR_POINTER;
  return forward_impl(x, logits, T, E, k, d, d_ff, w1_codes, w1_sf, w1_g, w2_codes, w2_sf, w2_g, out, ws, ws_bytes,
                      nullptr, nullptr, nullptr, false, status, stream, events);
}

int moe_expert_forward_gather(const uint16_t* x, const float* logits, int T, int E, int k, int d, int d_ff,
                              const uint8_t* w1_codes, const uint8_t* w1_sf, const float* w1_g,
                              const uint8_t* w2_codes, const uint8_t* w2_sf, const float* w2_g, uint16_t* out,
                              void* ws, size_t ws_bytes, int* status, void* stream) {
  // a code row of d/2 bytes must cover the 128-byte gather box
  if (d < 256) return MOE_ERR_SHAPE;
  return forward_impl(x, logits, T, E, k, d, d_ff, w1_codes, w1_sf, w1_g, w2_codes, w2_sf, w2_g, out, ws, ws_bytes,
                      nullptr, nullptr, nullptr, true, status, stream);
}

int moe_expert_forward_train(const uint16_t* x, const float* logits, int T, int E, int k, int d, int d_ff,
                             const uint8_t* w1_codes, const uint8_t* w1_sf, const float* w1_g,
                             const uint8_t* w2_codes, const uint8_t* w2_sf, const float* w2_g, uint16_t* out,
                             void* ws, size_t ws_bytes, uint16_t* save_u, uint16_t* save_h, int* status,
                             void* stream) {
  if (T > 0 && (!ok_ptr(save_u) || !ok_ptr(save_h))) return MOE_ERR_POINTER;
  return forward_impl(x, logits, T, E, k, d, d_ff, w1_codes, w1_sf, w1_g, w2_codes, w2_sf, w2_g, out, ws, ws_bytes,
                      save_u, save_h, nullptr, false, status, stream);
}

size_t moe_expert_backward_workspace_bytes(int T, int E, int k, int d, int d_ff) {
  if (!ok_model_shape(T, E, k, d, d_ff)) return 0;
  return bwd_layout(T, E, k, d, d_ff).total;
}

int moe_expert_backward(const uint16_t* dY, const uint16_t* x, int T, int E, int k, int d, int d_ff,
                        const uint16_t* W1, const uint16_t* W2, const uint8_t* w2_codes, const uint8_t* w2_sf,
                        const float* w2_g, const int32_t* topk_ids, const float* topk_w, const int32_t* offsets,
                        const int32_t* row_to_token, const int32_t* token_slot_row, const uint16_t* u,
                        const uint16_t* h, const uint8_t* h_codes, const uint8_t* h_sf, const float* h_g, float* dx,
                        float* dW1, float* dW2, float* dlogits, float* dw, void* ws, size_t ws_bytes, int* status,
                        void* stream) {
  if (!ok_model_shape(T, E, k, d, d_ff)) return MOE_ERR_SHAPE;
  if (!ok_ptr(W1) || !ok_ptr(W2) || !ok_ptr(dW1) || !ok_ptr(dW2) || !ok_opt(dlogits) || !ok_opt(status))
    return MOE_ERR_POINTER;
  if (T > 0 && (!ok_ptr(dY) || !ok_ptr(x) || !ok_ptr(w2_codes) || !ok_ptr(w2_sf) || !ok_ptr(w2_g) ||
                !ok_ptr(topk_ids) || !ok_ptr(topk_w) || !ok_ptr(offsets) || !ok_ptr(row_to_token) ||
                !ok_ptr(token_slot_row) || !ok_ptr(u) || !ok_ptr(h) || !ok_ptr(h_codes) || !ok_ptr(h_sf) ||
                !ok_ptr(h_g) || !ok_ptr(dx) || !ok_ptr(dw) || !ok_ptr(ws)))
    return MOE_ERR_POINTER;
  const BwdLayout L = bwd_layout(T, E, k, d, d_ff);
  if (T > 0 && ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  int rc = check_device();
  if (rc != MOE_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if (T == 0) {  // no rows: zero weight gradients
    if (cudaMemsetAsync(dW1, 0, (size_t)E * 2 * d_ff * d * 4, s) != cudaSuccess ||
        cudaMemsetAsync(dW2, 0, (size_t)E * d * d_ff * 4, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return finish();
  }
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* dy2 = reinterpret_cast<uint16_t*>(w + L.off[0]);
  uint16_t* xp = reinterpret_cast<uint16_t*>(w + L.off[1]);
  uint16_t* du = reinterpret_cast<uint16_t*>(w + L.off[2]);
  float* dxr = reinterpret_cast<float*>(w + L.off[3]);
  const int64_t mc = m_cap_of(T, E, k);
  const int F = d_ff;

  // the forward's FC2 again (same kernel, same y2), against dY: dw and dy2
  moe::Fc2Args a2;
  std::memset(&a2, 0, sizeof(a2));
  if (encode_operand(&a2.tmap_a, h_codes, mc, F / 2) != MOE_OK) return MOE_ERR_CUDA;
  if (encode_operand(&a2.tmap_b, w2_codes, (int64_t)E * d, F / 2) != MOE_OK) return MOE_ERR_CUDA;
  a2.a_sf = h_sf; a2.a_g = h_g; a2.w_sf = w2_sf; a2.w_g = w2_g; a2.offsets = offsets;
  a2.E = E; a2.d_ff = F; a2.d = d; a2.k = k;
  a2.row_to_token = row_to_token; a2.token_slot_row = token_slot_row; a2.topk_w = topk_w;
  a2.dY = dY; a2.dw = dw; a2.status = status;
  if (encode_bf16(&a2.tmap_out, dy2, mc, d, 32) != MOE_OK) return MOE_ERR_CUDA;
  if (moe::launch_fc2(a2, mc, s) != 0) return MOE_ERR_CUDA;
  if (dlogits) moe::launch_bwd_logits(dw, topk_w, topk_ids, T, E, k, dlogits, s);
  // The permuted x rows (read only by the dW1 GEMM) are copied on a second
  // stream, by one block per SM, beside the three GEMMs before dW1: both fit
  // on an SM together, and the copy's HBM traffic fills what the GEMMs leave.
  // (MOE_BWD_SIDE_STREAM=0 in the environment keeps it on the caller's stream.)
  const char* side_env = std::getenv("MOE_BWD_SIDE_STREAM");
  SideStream* side = nullptr;
  const bool forked = !(side_env && side_env[0] == '0') && side_stream(side) &&
                      cudaEventRecord(side->fork, s) == cudaSuccess &&
                      cudaStreamWaitEvent(side->s, side->fork, 0) == cudaSuccess;
  if (forked) {
    moe::launch_bwd_xrows(x, row_to_token, offsets, E, T, d, mc, xp, moe::gemm_num_ctas(), side->s);
    if (cudaEventRecord(side->join, side->s) != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    (void)cudaGetLastError();
    moe::launch_bwd_xrows(x, row_to_token, offsets, E, T, d, mc, xp, 0, s);
  }
  // an early return still leaves the caller's stream waiting for the copy
  auto fail = [&]() {
    if (forked) (void)cudaStreamWaitEvent(s, side->join, 0);
    return MOE_ERR_CUDA;
  };

  moe::BwdGemmArgs g;
  // dh = dy2 . W2_e, SwiGLU backward -> du
  std::memset(&g, 0, sizeof(g));
  if (encode_bf16(&g.tmap_a, dy2, mc, d, 128) != MOE_OK || encode_bf16(&g.tmap_b, W2, (int64_t)E * d, F, 64) != MOE_OK)
    return fail();
  g.mode = moe::BWD_DGRAD_SWIGLU; g.a_mn = 0; g.E = E; g.offsets = offsets; g.N = F; g.K = d; g.F = F;
  g.u = u; g.du = du; g.status = status;
  if (moe::launch_bwd_gemm(g, (int)(mc / 128), s) != 0) return fail();
  // dW2_e = dy2_e^T . h_e
  std::memset(&g, 0, sizeof(g));
  if (encode_bf16(&g.tmap_a, dy2, mc, d, 64) != MOE_OK || encode_bf16(&g.tmap_b, h, mc, F, 64) != MOE_OK)
    return fail();
  if (encode_f32_out(&g.tmap_out, dW2, (int64_t)E * d, F) != MOE_OK) return fail();
  g.mode = moe::BWD_WGRAD; g.a_mn = 1; g.E = E; g.offsets = offsets; g.N = F; g.Mo = d; g.out = dW2; g.status = status;
  if (moe::launch_bwd_gemm(g, 0, s) != 0) return fail();
  // dxr = du . W1_e
  std::memset(&g, 0, sizeof(g));
  if (encode_bf16(&g.tmap_a, du, mc, 2 * F, 128) != MOE_OK ||
      encode_bf16(&g.tmap_b, W1, (int64_t)E * 2 * F, d, 64) != MOE_OK)
    return fail();
  if (encode_f32_out(&g.tmap_out, dxr, mc, d) != MOE_OK) return fail();
  g.mode = moe::BWD_DGRAD; g.a_mn = 0; g.E = E; g.offsets = offsets; g.N = d; g.K = 2 * F; g.out = dxr;
  g.status = status;
  if (moe::launch_bwd_gemm(g, (int)(mc / 128), s) != 0) return fail();
  // dW1_e = du_e^T . xp_e
  if (forked && cudaStreamWaitEvent(s, side->join, 0) != cudaSuccess) return fail();
  std::memset(&g, 0, sizeof(g));
  if (encode_bf16(&g.tmap_a, du, mc, 2 * F, 64) != MOE_OK || encode_bf16(&g.tmap_b, xp, mc, d, 64) != MOE_OK)
    return fail();
  if (encode_f32_out(&g.tmap_out, dW1, (int64_t)E * 2 * F, d) != MOE_OK) return fail();
  g.mode = moe::BWD_WGRAD; g.a_mn = 1; g.E = E; g.offsets = offsets; g.N = d; g.Mo = 2 * F; g.out = dW1;
  g.status = status;
  if (moe::launch_bwd_gemm(g, 0, s) != 0) return fail();
  moe::launch_bwd_dx(dxr, token_slot_row, T, k, d, dx, s);
  return finish();
}

}  // extern "C"

namespace {

int forward_impl(const uint16_t* x, const float* logits, int T, int E, int k, int d, int d_ff,
                 const uint8_t* w1_codes, const uint8_t* w1_sf, const float* w1_g, const uint8_t* w2_codes,
                 const uint8_t* w2_sf, const float* w2_g, uint16_t* out, void* ws, size_t ws_bytes, uint16_t* save_u,
                 uint16_t* save_h, float* save_y2, bool gather, int* status, void* stream, void* const* events) {
  if (!ok_model_shape(T, E, k, d, d_ff)) return MOE_ERR_SHAPE;
  if (!ok_ptr(w1_codes) || !ok_ptr(w1_sf) || !ok_ptr(w1_g) || !ok_ptr(w2_codes) || !ok_ptr(w2_sf) || !ok_ptr(w2_g) ||
      !ok_opt(status))
    return MOE_ERR_POINTER;
  if (T > 0 && (!ok_ptr(x) || !ok_ptr(logits) || !ok_ptr(out) || !ok_ptr(ws))) return MOE_ERR_POINTER;
  const FwdLayout L = fwd_layout(T, E, k, d, d_ff);
  if (T > 0 && ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  int rc = check_device();
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* topk_ids = reinterpret_cast<int32_t*>(w + L.off[0]);
  float* topk_w = reinterpret_cast<float*>(w + L.off[1]);
  int32_t* tsr = reinterpret_cast<int32_t*>(w + L.off[2]);
  int32_t* counts = reinterpret_cast<int32_t*>(w + L.off[3]);
  int32_t* offsets = reinterpret_cast<int32_t*>(w + L.off[4]);
  int32_t* r2t = reinterpret_cast<int32_t*>(w + L.off[5]);
  float* amax_tok = reinterpret_cast<float*>(w + L.off[6]);
  uint8_t* x_codes = w + L.off[7];
  uint8_t* x_sf = w + L.off[8];
  float* x_g = reinterpret_cast<float*>(w + L.off[9]);
  uint8_t* h_codes = w + L.off[10];
  uint8_t* h_sf = w + L.off[11];
  float* h_g = reinterpret_cast<float*>(w + L.off[12]);
  uint16_t* slots = reinterpret_cast<uint16_t*>(w + L.off[13]);
  int32_t* hist = reinterpret_cast<int32_t*>(w + L.off[14]);
  uint16_t* scratch = reinterpret_cast<uint16_t*>(w + L.off[15]);
  const int64_t mc = m_cap_of(T, E, k);
  const int C = (T + kRouteChunk - 1) / kRouteChunk;
  // caller-owned events recorded before the first launch and after each
  auto mark = [&](int i) {
    if (events) (void)cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), s);
  };

  mark(0);
  moe::launch_route(logits, nullptr, nullptr, T, E, k, topk_ids, topk_w, tsr, hist, status, s);
  mark(1);
  moe::launch_scan(hist, C, E, counts, s);
  mark(2);
  // gather: x_codes holds the codes once per token (rows 0..T-1) and a zero
  // row T, which the pad rows gather; otherwise one copy per routed row
  moe::launch_pad_rows(offsets, counts, E, mc, r2t, nullptr, gather ? nullptr : x_codes, d, x_sf, x_g, s);
  mark(3);
  if (moe::launch_permute_quant(topk_ids, tsr, hist, offsets, T, E, k, x, d, r2t, amax_tok, gather ? nullptr : x_codes,
                                gather ? x_codes : nullptr, x_sf, x_g, status, s) != 0)
    return MOE_ERR_CUDA;
  mark(4);

  moe::Fc1Args a1;
  std::memset(&a1, 0, sizeof(a1));
  if (gather) {
    if (encode_gather_rows(&a1.tmap_a, x_codes, (int64_t)T + 1, d / 2) != MOE_OK) return MOE_ERR_CUDA;
    a1.a_rows = r2t;
    a1.zero_row = T;
  } else if (encode_operand(&a1.tmap_a, x_codes, mc, d / 2) != MOE_OK) {
    return MOE_ERR_CUDA;
  }
  if (encode_operand(&a1.tmap_b, w1_codes, (int64_t)E * 2 * d_ff, d / 2) != MOE_OK) return MOE_ERR_CUDA;
  a1.a_sf = x_sf; a1.a_g = x_g; a1.w_sf = w1_sf; a1.w_g = w1_g; a1.offsets = offsets;
  a1.E = E; a1.d = d; a1.d_ff = d_ff;
  a1.h_codes = h_codes; a1.h_sf = h_sf; a1.h_g = h_g; a1.scratch = scratch; a1.status = status;
  a1.save_u = save_u; a1.dbg_h = save_h;
  if (moe::launch_fc1(a1, mc, s) != 0) return MOE_ERR_CUDA;
  mark(5);

  moe::Fc2Args a2;
  std::memset(&a2, 0, sizeof(a2));
  if (encode_operand(&a2.tmap_a, h_codes, mc, d_ff / 2) != MOE_OK) return MOE_ERR_CUDA;
  if (encode_operand(&a2.tmap_b, w2_codes, (int64_t)E * d, d_ff / 2) != MOE_OK) return MOE_ERR_CUDA;
  a2.a_sf = h_sf; a2.a_g = h_g; a2.w_sf = w2_sf; a2.w_g = w2_g; a2.offsets = offsets;
  a2.E = E; a2.d_ff = d_ff; a2.d = d; a2.k = k;
  a2.row_to_token = r2t; a2.token_slot_row = tsr; a2.topk_w = topk_w; a2.status = status;
  a2.dbg_y = save_y2;
  if (encode_bf16(&a2.tmap_out, slots, mc, d, 32) != MOE_OK) return MOE_ERR_CUDA;
  if (moe::launch_fc2(a2, mc, s) != 0) return MOE_ERR_CUDA;
  mark(6);
  moe::launch_unpermute_reduce(slots, tsr, T, k, d, out, s);
  mark(7);
  return finish();
}

}  // namespace
