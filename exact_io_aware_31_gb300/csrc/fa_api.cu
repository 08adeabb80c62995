// The C ABI of include/fa.h: argument validation, TMA tensor maps, the device
// status word, and kernel launches.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "fa_common.cuh"
#include "fa_context.h"
#include "fa_kernels.h"

namespace fa {

// One status word per device that loads this library.  Kernels write
// FA_ERR_DEVICE_TIMEOUT here when a bounded wait gives up.
__device__ int g_device_status;

namespace {

constexpr int kMaxDevices = 64;

// Facts about the current device plus the status word's address in the
// current context.
struct DeviceInfo {
  int sms = 0;
  bool sm103 = false;
  int* status = nullptr;  // device address of g_device_status in the current context
};

struct DeviceProps {
  bool ready = false;
  int sms = 0;
  bool sm103 = false;
};

std::mutex g_mu;
DeviceProps g_dev[kMaxDevices];
PerContextAddress g_status_addr;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Device properties are resolved once per device; the status word's address
// once per context (a device address is only valid in the context that gave
// it).
int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceProps& d = g_dev[dev];
    if (!d.ready) {
      int major = 0, minor = 0, sms = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
      }
      if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
          cudaGetLastError();
          return FA_ERR_CUDA;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
      d.sm103 = (major == 10 && minor == 3);
      d.sms = sms;
      d.ready = true;
    }
    out->sms = d.sms;
    out->sm103 = d.sm103;
  }
  if (!out->sm103) return FA_ERR_UNSUPPORTED;
  void* p = nullptr;
  if (g_status_addr.get(&p, [](void** q) { return cudaGetSymbolAddress(q, g_device_status); }) != 0)
    return FA_ERR_CUDA;
  out->status = static_cast<int*>(p);
  return FA_OK;
}

// [B*H, N, d] bf16 viewed as a 3-D tensor; box_rows-row x 64-column boxes
// (128 unless given), 128-byte swizzle (the layout the tcgen05 descriptors
// expect).
int make_map(CUtensorMap* m, const void* base, int BH, int N, int d, unsigned box_rows = 128) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// [B*H, N, d] fp32 (the dQ accumulator): 128-row x 32-column boxes,
// 128-byte swizzle, used by the tensor reduce-add of the d = 64 backward.
int make_map_f32(CUtensorMap* m, const void* base, int BH, int N, int d) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// [B*H, N, d] E4M3 codes (one byte each) for the FP8 forward, d = 128: one
// 128-row x 128-column box is one 128-byte-swizzled block.
int make_map_e4m3(CUtensorMap* m, const void* base, int BH, int N, int d) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)N * d};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_sizes(int B, int H, int N, int d, float scale, int causal) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  if (bh > INT_MAX || (long long)N > (1 << 30)) return FA_ERR_INVALID_ARG;
  const long long npad = ((long long)N + 127) / 128 * 128;
  if (bh * npad * (d > 0 ? d : 1) >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// scale * log2(e), its magnitude floored at 1e-30 so that a masked score
// (-inf) times |c2| stays -inf when scale == 0.  For finite scores |s| < 1e8
// the floor changes 2^(s * c2) by less than one fp32 ulp of 1, so scale == 0
// still gives exact uniform attention.  The sign is kept: the tensor-core
// kernels compute S negated for a negative scale and use |c2| after it.
float log2_scale(float scale) {
  const float c2 = scale * 1.4426950408889634f;
  return std::fabs(c2) > 1e-30f ? c2 : std::copysign(1e-30f, c2);
}

struct WorkspaceLayout {
  size_t dq_acc, lse2, dsum, total;
};

WorkspaceLayout workspace_layout(int B, int H, int N, int d) {
  const size_t bh = (size_t)B * H;
  const size_t npad = ((size_t)N + 127) / 128 * 128;
  WorkspaceLayout w;
  w.dq_acc = 0;
  w.lse2 = round256(bh * (size_t)N * d * 4);
  w.dsum = w.lse2 + round256(bh * npad * 4);
  w.total = w.dsum + round256(bh * npad * 4);
  return w;
}

// The forward's launch once the arguments are validated and the tensor maps
// built (shared by fa_fwd, fa_fwd_fp8 and fa_fwd_dropout).  c2 = scale (times
// the FP8 descale factors) * log2(e); `drop` is used when dropout != 0.
int run_forward(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, void* o, float* lse, int BH,
                int N, int d, int causal, float c2, const DeviceInfo& dev, int fp8, int dropout, const DropParams& drop,
                cudaStream_t stream) {
  FwdLaunch a;
  // The output in 32-row boxes, one per softmax warp, for the kernels that
  // store O with TMA (d = 64, N < 4096); the others never read the map.
  CUtensorMap to;
  const bool o_map = d == 64 && !fp8 && N < 4096;
  if (o_map && make_map(&to, o, BH, N, d, 32)) return FA_ERR_CUDA;
  a.tm_q = &tq;
  a.tm_k = &tk;
  a.tm_v = &tv;
  a.tm_o = o_map ? &to : &tq;
  a.o = o;
  a.lse = lse;
  a.BH = BH;
  a.N = N;
  a.d = d;
  a.causal = causal;
  a.c2 = c2;
  a.status = dev.status;
  a.fp8 = fp8;
  a.dropout = dropout;
  a.drop = drop;
  const int units = fwd_units(BH, N);
  a.grid = units < dev.sms ? units : dev.sms;
  if (launch_fwd(a, stream) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                      float scale, int causal, cudaStream_t stream) {
  int st = check_sizes(B, H, N, d, scale, causal);
  if (st != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FA_OK) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if (make_map(&tq, q, BH, N, d) || make_map(&tk, k, BH, N, d) || make_map(&tv, v, BH, N, d)) return FA_ERR_CUDA;
  return run_forward(tq, tk, tv, o, lse, BH, N, d, causal, log2_scale(scale), dev, 0, 0, DropParams{}, stream);
}

extern "C" int fa_fwd_fp8(const void* q8, const void* k8, const void* v, void* o, float* lse, int B, int H, int N,
                          int d, float scale, float q_descale, float k_descale, int causal, cudaStream_t stream) {
  int st = check_sizes(B, H, N, d, scale, causal);
  if (st != FA_OK) return st;
  if (!std::isfinite(q_descale) || !std::isfinite(k_descale) || q_descale < 0.f || k_descale < 0.f || scale < 0.f)
    return FA_ERR_INVALID_ARG;
  const float eff = scale * q_descale * k_descale;
  if (!std::isfinite(eff)) return FA_ERR_INVALID_ARG;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FA_OK) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if (make_map_e4m3(&tq, q8, BH, N, d) || make_map_e4m3(&tk, k8, BH, N, d) || make_map(&tv, v, BH, N, d))
    return FA_ERR_CUDA;
  return run_forward(tq, tk, tv, o, lse, BH, N, d, causal, log2_scale(eff), dev, 1, 0, DropParams{}, stream);
}

namespace fa {
namespace {

constexpr int kMaxDecodeQueries = 8;

int check_decode(int B, int H, int Nq, int Nk, int d, float scale, int causal, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || num_splits < 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  if (bh > INT_MAX || (long long)Nk > (1 << 30)) return FA_ERR_INVALID_ARG;
  const long long kpad = ((long long)Nk + 127) / 128 * 128;
  if (bh * kpad * (d > 0 ? d : 1) >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return FA_ERR_INVALID_ARG;  // a query would see no key
  if (Nq > kMaxDecodeQueries) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Clusters of `size` decode split CTAs the device can hold at once, for both
// masks (the smaller count); asked once per (device, d, query bucket, size).
int decode_cluster_capacity(int dev, int d, int Nq, int size) {
  if (size < 2 || size > 16) return 0;
  static std::mutex mu;
  static int known[kMaxDevices][2][4][17];  // capacity + 1; 0 = not asked yet
  const int qb = Nq <= 1 ? 0 : Nq <= 2 ? 1 : Nq <= 4 ? 2 : 3;
  std::lock_guard<std::mutex> lock(mu);
  int& k = known[dev][d == 128][qb][size];
  if (k == 0) {
    const int a = decode_max_clusters(d, Nq, 0, size), b = decode_max_clusters(d, Nq, 1, size);
    k = (a < b ? a : b) + 1;
  }
  return k - 1;
}

// Splits per head and whether they merge inside one cluster.  The requested
// number (never more than the 128-key tiles), or (0) as many as fill the SMs
// with one CTA each.  A head's splits run as one cluster when every head's
// cluster fits on the device at once; the automatic choice takes down to 80%
// of its split count to get there (the cluster merge saves the second kernel
// and its launch gap).  Otherwise the splits merge through the workspace.
int decode_plan(int dev, long long bh, int Nq, int Nk, int d, int num_splits, int sms, bool* cluster) {
  const int tiles = (Nk + 127) / 128;
  *cluster = false;
  if (num_splits > 0) {
    const int s = num_splits < tiles ? num_splits : tiles;
    *cluster = s >= 2 && decode_cluster_capacity(dev, d, Nq, s) >= bh;
    return s;
  }
  long long s0 = sms / bh > 1 ? sms / bh : 1;
  if (s0 > tiles) s0 = tiles;
  if (s0 < 2) return (int)s0;
  const int lo = (int)((4 * s0 + 4) / 5) > 2 ? (int)((4 * s0 + 4) / 5) : 2;
  for (int s = (int)(s0 < 16 ? s0 : 16); s >= lo; --s)
    if (decode_cluster_capacity(dev, d, Nq, s) >= bh) {
      *cluster = true;
      return s;
    }
  return (int)s0;
}

size_t decode_partials_bytes(long long bh, int Nq, int d, int splits, bool cluster) {
  if (splits <= 1 || cluster) return 0;
  return round256((size_t)splits * bh * Nq * d * 4) + round256((size_t)splits * bh * Nq * 4);
}

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return dev;
}

}  // namespace
}  // namespace fa

extern "C" size_t fa_fwd_splitkv_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (check_decode(B, H, Nq, Nk, d, 1.0f, 0, num_splits) != FA_OK) return 0;
  DeviceInfo dev;
  if (device_info(&dev) != FA_OK) return 0;
  const long long bh = (long long)B * H;
  bool cluster = false;
  const int splits = decode_plan(current_device(), bh, Nq, Nk, d, num_splits, dev.sms, &cluster);
  return decode_partials_bytes(bh, Nq, d, splits, cluster);
}

extern "C" int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                              int Nk, int d, float scale, int causal, int num_splits, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  int st = check_decode(B, H, Nq, Nk, d, scale, causal, num_splits);
  if (st != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FA_OK) return st;
  const int BH = B * H;
  DecLaunch a;
  bool cluster = false;
  a.splits = decode_plan(current_device(), BH, Nq, Nk, d, num_splits, dev.sms, &cluster);
  a.cluster = cluster ? 1 : 0;
  const size_t need = decode_partials_bytes(BH, Nq, d, a.splits, cluster);
  if (need > 0 && (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                   workspace_bytes < need))
    return FA_ERR_WORKSPACE;
  CUtensorMap tq, tk, tv;
  if (make_map(&tq, q, BH, Nq, d) || make_map(&tk, k, BH, Nk, d) || make_map(&tv, v, BH, Nk, d)) return FA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.tm_q = &tq;
  a.tm_k = &tk;
  a.tm_v = &tv;
  a.q = q;
  a.o = o;
  a.lse = lse;
  a.part_o = need ? reinterpret_cast<float*>(ws) : nullptr;
  a.part_lse2 = need ? reinterpret_cast<float*>(ws + round256((size_t)a.splits * BH * Nq * d * 4)) : nullptr;
  a.BH = BH;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.causal = causal;
  a.c2 = log2_scale(scale);
  a.status = dev.status;
  if (launch_decode(a, stream) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

namespace fa {
namespace {

// Dropout parameters of the C ABI -> kernel form; FA_ERR_INVALID_ARG unless 0 <= p < 1.
int drop_params(float p_drop, unsigned long long seed, unsigned int offset, DropParams* out) {
  if (!std::isfinite(p_drop) || p_drop < 0.f || p_drop >= 1.f) return FA_ERR_INVALID_ARG;
  const double t = std::nearbyint((double)p_drop * 4294967296.0);
  out->thr = t >= 4294967295.0 ? 0xFFFFFFFFu : (uint32_t)t;
  out->k0 = (uint32_t)(seed & 0xFFFFFFFFull);
  out->k1 = (uint32_t)(seed >> 32);
  out->offset = offset;
  out->inv_keep = (float)(1.0 / (1.0 - (double)p_drop));
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" int fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                              int d, float scale, int causal, float p_drop, unsigned long long seed,
                              unsigned int offset, cudaStream_t stream) {
  DropParams dp;
  int st = drop_params(p_drop, seed, offset, &dp);
  if (st != FA_OK) return st;
  if ((st = check_sizes(B, H, N, d, scale, causal)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FA_OK) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if (make_map(&tq, q, BH, N, d) || make_map(&tk, k, BH, N, d) || make_map(&tv, v, BH, N, d)) return FA_ERR_CUDA;
  return run_forward(tq, tk, tv, o, lse, BH, N, d, causal, log2_scale(scale), dev, 0, 1, dp, stream);
}

extern "C" size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (check_sizes(B, H, N, d, 1.0f, 0) != FA_OK) return 0;
  return workspace_layout(B, H, N, d).total;
}

namespace fa {
namespace {

// Validation and launch arguments shared by fa_bwd and its three phases.
// `need` selects which tensor pointers the caller must supply.
enum : unsigned { kNeedQKV = 1, kNeedO = 2, kNeedDout = 4, kNeedLse = 8, kNeedDq = 16, kNeedDkDv = 32 };

int prepare_bwd(BwdLaunch& a, CUtensorMap* maps, unsigned need, const void* q, const void* k, const void* v,
                const void* o, const void* dout, const float* lse, void* dq, void* dk, void* dv, int B, int H, int N,
                int d, float scale, int causal, const void* workspace, size_t workspace_bytes) {
  int st = check_sizes(B, H, N, d, scale, causal);
  if (st != FA_OK) return st;
  if (((need & kNeedQKV) && (!aligned16(q) || !aligned16(k) || !aligned16(v))) ||
      ((need & kNeedO) && !aligned16(o)) || ((need & kNeedDout) && !aligned16(dout)) ||
      ((need & kNeedLse) && !aligned16(lse)) || ((need & kNeedDq) && !aligned16(dq)) ||
      ((need & kNeedDkDv) && (!aligned16(dk) || !aligned16(dv))))
    return FA_ERR_INVALID_ARG;
  const WorkspaceLayout w = workspace_layout(B, H, N, d);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < w.total)
    return FA_ERR_WORKSPACE;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FA_OK) return st;
  const int BH = B * H;
  if (need & kNeedQKV) {
    if (make_map(&maps[0], q, BH, N, d) || make_map(&maps[1], k, BH, N, d) || make_map(&maps[2], v, BH, N, d) ||
        make_map(&maps[3], dout, BH, N, d))
      return FA_ERR_CUDA;
  }
  uint8_t* ws = static_cast<uint8_t*>(const_cast<void*>(workspace));
  if ((need & kNeedQKV) && make_map_f32(&maps[4], ws + w.dq_acc, BH, N, d)) return FA_ERR_CUDA;
  if ((need & kNeedDkDv) && (make_map(&maps[5], dk, BH, N, d) || make_map(&maps[6], dv, BH, N, d)))
    return FA_ERR_CUDA;
  a.tm_dqacc = &maps[4];
  a.tm_dk = &maps[5];
  a.tm_dv = &maps[6];
  a.tm_q = &maps[0];
  a.tm_k = &maps[1];
  a.tm_v = &maps[2];
  a.tm_do = &maps[3];
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dq_acc = reinterpret_cast<float*>(ws + w.dq_acc);
  a.lse2 = reinterpret_cast<float*>(ws + w.lse2);
  a.dsum = reinterpret_cast<float*>(ws + w.dsum);
  a.BH = BH;
  a.N = N;
  a.Npad = (N + 127) / 128 * 128;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  a.c2 = log2_scale(scale);
  a.status = dev.status;
  const int units = bwd_units(BH, N);
  a.grid = units < dev.sms ? units : dev.sms;
  a.pre_grid = dev.sms * 8;
  return FA_OK;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FA_OK;
  cudaGetLastError();
  return FA_ERR_CUDA;
}

}  // namespace
}  // namespace fa

extern "C" int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                      void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  BwdLaunch a;
  CUtensorMap maps[7];
  int st = prepare_bwd(a, maps, kNeedQKV | kNeedO | kNeedDout | kNeedLse | kNeedDq | kNeedDkDv, q, k, v, o, dout,
                       lse, dq, dk, dv, B, H, N, d, scale, causal, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  if ((st = cuda_status(launch_bwd_pre(a, stream))) != FA_OK) return st;
  if ((st = cuda_status(launch_bwd_main(a, stream))) != FA_OK) return st;
  return cuda_status(launch_bwd_conv(a, stream));
}

extern "C" int fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                              int causal, float p_drop, unsigned long long seed, unsigned int offset,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  DropParams dp;
  int st = drop_params(p_drop, seed, offset, &dp);
  if (st != FA_OK) return st;
  BwdLaunch a;
  CUtensorMap maps[7];
  st = prepare_bwd(a, maps, kNeedQKV | kNeedO | kNeedDout | kNeedLse | kNeedDq | kNeedDkDv, q, k, v, o, dout, lse, dq,
                   dk, dv, B, H, N, d, scale, causal, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  a.dropout = 1;
  a.drop = dp;
  if ((st = cuda_status(launch_bwd_pre(a, stream))) != FA_OK) return st;
  if ((st = cuda_status(launch_bwd_main(a, stream))) != FA_OK) return st;
  return cuda_status(launch_bwd_conv(a, stream));
}

extern "C" int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                    const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                    float scale, int causal, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
  BwdLaunch a;
  CUtensorMap maps[7];
  int st = prepare_bwd(a, maps, kNeedQKV | kNeedO | kNeedDout | kNeedLse | kNeedDq | kNeedDkDv, q, k, v, o, dout,
                       lse, dq, dk, dv, B, H, N, d, scale, causal, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  a.with_dq = 0;  // dK / dV kernel without dQ; dQ from the query-outer kernel
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FA_OK) return st;
  const int units = bwd_dq_units(a.BH, N);
  a.dq_grid = units < dev.sms ? units : dev.sms;
  if ((st = cuda_status(launch_bwd_pre(a, stream))) != FA_OK) return st;
  if ((st = cuda_status(launch_bwd_main(a, stream))) != FA_OK) return st;
  return cuda_status(launch_bwd_dq(a, stream));
}

extern "C" int fa_bwd_preprocess(const void* o, const void* dout, const float* lse, int B, int H, int N, int d,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  BwdLaunch a;
  CUtensorMap maps[7];
  int st = prepare_bwd(a, maps, kNeedO | kNeedDout | kNeedLse, nullptr, nullptr, nullptr, o, dout, lse, nullptr,
                       nullptr, nullptr, B, H, N, d, 1.0f, 0, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  return cuda_status(launch_bwd_pre(a, stream));
}

extern "C" int fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv, int B,
                           int H, int N, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  BwdLaunch a;
  CUtensorMap maps[7];
  int st = prepare_bwd(a, maps, kNeedQKV | kNeedDout | kNeedDkDv, q, k, v, nullptr, dout, nullptr, nullptr, dk, dv,
                       B, H, N, d, scale, causal, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  return cuda_status(launch_bwd_main(a, stream));
}

extern "C" int fa_bwd_dq_convert(void* dq, int B, int H, int N, int d, float scale, const void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
  BwdLaunch a;
  CUtensorMap maps[7];
  int st = prepare_bwd(a, maps, kNeedDq, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dq, nullptr, nullptr,
                       B, H, N, d, scale, 0, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  return cuda_status(launch_bwd_conv(a, stream));
}

extern "C" int fa_get_device_status(cudaStream_t stream) {
  DeviceInfo dev;
  int st = device_info(&dev);
  if (st != FA_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  int value = 0, zero = 0;
  if (cudaMemcpy(&value, dev.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(dev.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return value;
}

extern "C" const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK:
      return "FA_OK";
    case FA_ERR_INVALID_ARG:
      return "FA_ERR_INVALID_ARG: invalid pointer, size, scale or mask flag";
    case FA_ERR_UNSUPPORTED:
      return "FA_ERR_UNSUPPORTED: head dimension must be 64 or 128 on an sm_103 device";
    case FA_ERR_WORKSPACE:
      return "FA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case FA_ERR_CUDA:
      return "FA_ERR_CUDA: a CUDA call or kernel launch failed";
    case FA_ERR_DEVICE_TIMEOUT:
      return "FA_ERR_DEVICE_TIMEOUT: a kernel gave up on a bounded wait";
    case FA_ERR_INTERNAL:
      return "FA_ERR_INTERNAL: a kernel found an internal layout assumption violated";
    default:
      return "unknown fa status";
  }
}
