// C ABI of libcbr.so: argument validation, workspace layout, tensor-map encoding and the
// ordering of the kernel launches for each public call (declared in include/cbr.h).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <set>
#include <utility>

#include "../../include/cbr.h"
#include "cbr_internal.h"

namespace cbr {

// Device error word: kernels OR failure bits into it instead of trapping.
__device__ uint32_t g_error_word;

namespace {

constexpr size_t kHdrBytes = kWsHeaderBytes;  // arrival counters live here
// header words: 0 the forward's finalize ticket, 1 the backward's, kReadyWord the persistent
// forward's ready word
constexpr int kReadyWord = 8;
constexpr int kMaxDevices = 64;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct DeviceInfo {
  bool probed = false;
  bool ok = false;
  int num_sms = 0;
  uint32_t* err = nullptr;
};
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Returns CBR status; fills *info for the current device.
int current_device(DeviceInfo** info) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return CBR_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    d.probed = true;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return CBR_ERR_DEVICE;
    }
    void* p = nullptr;
    if (major == 10 && minor == 3 && cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) {
      d.ok = true;
      d.num_sms = sms < kMaxCtas ? sms : kMaxCtas;
      d.err = static_cast<uint32_t*>(p);
    }
    cudaGetLastError();
  }
  if (!d.ok) return CBR_ERR_DEVICE;
  *info = &d;
  return CBR_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// ----------------------------------------------------------------------- profiling hook
thread_local void* const* t_prof_events = nullptr;
thread_local int t_prof_count = 0;
thread_local int t_prof_used = 0;

struct Prof {
  void* const* ev;
  int count;
  int used = 0;
  cudaStream_t st;
  Prof(cudaStream_t s) : ev(t_prof_events), count(t_prof_count), st(s) {
    t_prof_events = nullptr;
    t_prof_count = 0;
    mark();
  }
  // Under stream capture a plain event record only orders streams; the external flag makes
  // it a timestamping event-record node of the graph.
  void mark() {
    if (!ev || used >= count) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
      cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev[used++]), st, cudaEventRecordExternal);
    else
      cudaEventRecord(static_cast<cudaEvent_t>(ev[used++]), st);
  }
  ~Prof() { t_prof_used = used; }
};

// ----------------------------------------------------------------------- validation helpers
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Shape {
  long long n, h, w, cin, cout, r, s, stride, pad, p, q, m;
  bool bf16;
  size_t elt;
};

int check_desc(const cbr_desc_t* d, Shape* sh) {
  if (!d) return CBR_ERR_INVALID_ARG;
  if (d->n < 1 || d->h < 1 || d->w < 1 || d->c_in < 1 || d->c_out < 1 || d->r < 1 || d->s < 1 ||
      d->stride < 1 || d->pad < 0)
    return CBR_ERR_INVALID_ARG;
  if (d->dtype != CBR_F16 && d->dtype != CBR_BF16) return CBR_ERR_UNSUPPORTED;
  if (d->c_out % 8 != 0) return CBR_ERR_INVALID_ARG;
  Shape s;
  s.n = d->n; s.h = d->h; s.w = d->w; s.cin = d->c_in; s.cout = d->c_out;
  s.r = d->r; s.s = d->s; s.stride = d->stride; s.pad = d->pad;
  if (s.h + 2 * s.pad < s.r || s.w + 2 * s.pad < s.s) return CBR_ERR_INVALID_ARG;
  s.p = (s.h + 2 * s.pad - s.r) / s.stride + 1;
  s.q = (s.w + 2 * s.pad - s.s) / s.stride + 1;
  s.m = s.n * s.p * s.q;
  if (s.m < 2) return CBR_ERR_INVALID_ARG;
  s.bf16 = d->dtype == CBR_BF16;
  s.elt = 2;
  *sh = s;
  return CBR_OK;
}

bool is_first_layer(const Shape& s) { return s.cin == 3; }

// Shapes the library runs on the device.
int check_supported(const Shape& s) {
  if (!(s.cout == 16 || s.cout == 32 || s.cout == 64 || s.cout == 128)) return CBR_ERR_UNSUPPORTED;
  // first layer (3 channels): im2col kernels, any stride, filters up to 8x8, rows up to 128
  if (is_first_layer(s)) return (s.r <= 8 && s.s <= 8 && s.q <= 128) ? CBR_OK : CBR_ERR_UNSUPPORTED;
  if (s.stride != 1) return CBR_ERR_UNSUPPORTED;
  if (s.cin % 8 != 0 || s.cin > 128) return CBR_ERR_UNSUPPORTED;
  if (s.w + 2 * s.pad > 256) return CBR_ERR_UNSUPPORTED;
  return CBR_OK;
}

size_t act_bytes(long long n, long long h, long long w, long long c, size_t elt) {
  return (size_t)n * h * w * c * elt;
}

// Workspace layouts (offsets from ws).
struct FwdWs {
  size_t eq, part, z, total;
};
FwdWs fwd_ws(const Shape& s, bool need_z) {
  FwdWs L;
  L.eq = kHdrBytes;
  L.part = align_up(L.eq + 2 * s.cout * sizeof(float), 256);
  L.z = align_up(L.part + fprop_partial_floats(kMaxCtas, (int)s.cout) * sizeof(float), 256);
  L.total = need_z ? align_up(L.z + act_bytes(s.n, s.p, s.q, s.cout, s.elt), 256) : L.z;
  return L;
}
// Whether the fused backward kernel (dz evaluated on chip, both convolutions in one kernel)
// takes this layer; the other layers materialise dz once in the workspace.
bool use_fused_bwd(const Shape& s) {
  return !is_first_layer(s) && bwd_fused_supported((int)s.n, (int)s.h, (int)s.w, (int)s.cin, (int)s.cout,
                                                   (int)s.r, (int)s.s, (int)s.stride, (int)s.pad);
}

// Row pitch (pixels) of the materialised dz.  The halo convolutions read it in their
// padded-linear row space (pitch w + 2*pad, the columns past q zero), so a unit's dz tile is
// one contiguous run of rows; the first layer's wgrad reads plain [n][p][q] rows.
long long dz_pitch(const Shape& s) { return is_first_layer(s) ? s.q : s.w + 2 * s.pad; }

// Whether dz can be materialised: the padded dz kernel indexes vectors in 32 bits.
bool dz_materialisable(const Shape& s) {
  return is_first_layer(s) || s.n * s.p * dz_pitch(s) * (s.cout / 8) < (1ll << 31);
}

struct BwdWs {
  size_t coef, mbits, part, wpart, dz, z, total;
};
BwdWs bwd_ws(const Shape& s, bool need_z) {
  BwdWs L;
  L.coef = kHdrBytes;
  // the bit-packed form of a byte-per-element mask (CBR_MASK_BYTES), one bit per element
  L.mbits = align_up(L.coef + 3 * s.cout * sizeof(float), 256);
  L.part = align_up(L.mbits + (size_t)((s.m * s.cout + 31) / 32) * 4, 256);
  L.wpart = align_up(L.part + bwd_reduce_partial_floats(kMaxCtas, (int)s.cout) * sizeof(float), 256);
  const size_t wpart = is_first_layer(s) ? first_wgrad_partial_floats(kMaxCtas, (int)s.cout)
                                         : wgrad_partial_floats(kMaxCtas, (int)s.cin, (int)s.cout, (int)(s.r * s.s));
  L.dz = align_up(L.wpart + wpart * sizeof(float), 256);
  // materialised dz (none when the fused kernel evaluates it on chip)
  const size_t dz_bytes = use_fused_bwd(s) ? 0 : act_bytes(s.n, s.p, dz_pitch(s), s.cout, s.elt);
  L.z = align_up(L.dz + dz_bytes, 256);
  L.total = need_z ? align_up(L.z + act_bytes(s.n, s.p, s.q, s.cout, s.elt), 256) : L.z;
  return L;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

HaloGeom make_geom(const Shape& s) {
  HaloGeom g{};
  g.n_img = (int)s.n;
  g.h = (int)s.h;
  g.w = (int)s.w;
  g.r = (int)s.r;
  g.s = (int)s.s;
  g.pad = (int)s.pad;
  return g;
}

// Forward convolution of either family (halo tiling, or the first-layer im2col kernel).
int run_fprop(const FpropArgs& a, const Shape& s, const void* x, const void* w, int num_sms, cudaStream_t st) {
  if (is_first_layer(s)) return launch_first_fprop(a, (int)s.stride, (int)s.cout, s.bf16, x, w, num_sms, st);
  return launch_fprop(a, (int)s.cin, (int)s.cout, s.bf16, x, w, num_sms, st);
}

}  // namespace

namespace {
bool encode_tiled_mode(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swz);
}  // namespace

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tiled_mode(map, dt, rank, base, dims, strides_bytes, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool encode_tiled_plain(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tiled_mode(map, dt, rank, base, dims, strides_bytes, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool encode_tiled_span(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       int swizzle_bytes) {
  const CUtensorMapSwizzle swz = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                 : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                       : CU_TENSOR_MAP_SWIZZLE_NONE;
  return encode_tiled_mode(map, dt, rank, base, dims, strides_bytes, box, swz);
}

namespace {
bool encode_tiled_mode(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swz) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cudaGetLastError();
  });
  if (!g_encode) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  return g_encode(map, dt, (cuuint32_t)rank, const_cast<void*>(base), d, st, b, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

int check_forward_train(const void* desc, const void* x, const void* w, const float* gamma,
                        const float* beta, const float* running_mean, const float* running_var,
                        float momentum, float eps, const void* y, const uint32_t* relu_mask,
                        const void* z_saved, const float* saved_mean, const float* saved_inv_var,
                        size_t* ws_need) {
  Shape s;
  int st = check_desc(static_cast<const cbr_desc_t*>(desc), &s);
  if (st) return st;
  if (!x || !w || !gamma || !beta || !running_mean || !running_var || !y || !saved_mean ||
      !saved_inv_var)
    return CBR_ERR_INVALID_ARG;
  if (!(momentum >= 0.f && momentum <= 1.f) || !(eps > 0.f) || !std::isfinite(eps))
    return CBR_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || (z_saved && !aligned(z_saved, 16)) ||
      (relu_mask && !aligned(relu_mask, 4)) || !aligned(gamma, 4) || !aligned(beta, 4) ||
      !aligned(running_mean, 4) || !aligned(running_var, 4) || !aligned(saved_mean, 4) ||
      !aligned(saved_inv_var, 4))
    return CBR_ERR_MISALIGNED;
  if ((st = check_supported(s))) return st;
  *ws_need = fwd_ws(s, z_saved == nullptr).total;
  return CBR_OK;
}

int check_device() {
  DeviceInfo* dev = nullptr;
  return current_device(&dev);
}

bool ensure_smem_attr(const void* func, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(mu);
  if (done.count({dev, func})) return true;
  // the opt-in limit covers static and dynamic shared memory together: clamp to what is left
  // beside the kernel's static shared memory
  int optin = 0;
  cudaFuncAttributes fa{};
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, func) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  bytes = std::min(bytes, optin - (int)fa.sharedSizeBytes);
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();  // do not leave the failure for the next launch check to find
    return false;
  }
  done.insert({dev, func});
  return true;
}

int launch_fold(const void* w, const float* conv_bias, const float* gamma, const float* beta,
                const float* rm, const float* rv, float eps, void* w_fold, float* b_fold, int cout,
                int rsc, bool bf16, cudaStream_t st);

}  // namespace cbr

using namespace cbr;

extern "C" {

int32_t cbr_version(void) { return 100; }

const char* cbr_status_string(cbr_status_t s) {
  switch (s) {
    case CBR_OK: return "CBR_OK";
    case CBR_ERR_INVALID_ARG: return "CBR_ERR_INVALID_ARG";
    case CBR_ERR_MISALIGNED: return "CBR_ERR_MISALIGNED";
    case CBR_ERR_UNSUPPORTED: return "CBR_ERR_UNSUPPORTED";
    case CBR_ERR_WORKSPACE: return "CBR_ERR_WORKSPACE";
    case CBR_ERR_DEVICE: return "CBR_ERR_DEVICE";
    case CBR_ERR_CUDA: return "CBR_ERR_CUDA";
    case CBR_ERR_TIMEOUT: return "CBR_ERR_TIMEOUT";
  }
  return "CBR_ERR_UNKNOWN";
}

cbr_status_t cbr_workspace_size(const cbr_desc_t* desc, size_t* fwd_bytes, size_t* bwd_bytes) {
  Shape s;
  int st = check_desc(desc, &s);
  if (st) return (cbr_status_t)st;
  if (fwd_bytes) *fwd_bytes = fwd_ws(s, true).total;
  if (bwd_bytes) *bwd_bytes = bwd_ws(s, true).total;
  return CBR_OK;
}

}  // extern "C"

namespace {

// The training forward; persistent: the one-launch form (conv, statistics, finalize and apply in
// one cooperative kernel), or CBR_ERR_UNSUPPORTED where the batch's accumulators do not all fit
// in TMEM at once.
cbr_status_t forward_train_impl(bool persistent, const cbr_desc_t* desc, const void* x, const void* w,
                                const float* gamma, const float* beta, float* running_mean, float* running_var,
                                float momentum, float eps, void* y, uint32_t* relu_mask, void* z_saved,
                                float* saved_mean, float* saved_inv_var, void* ws, size_t ws_bytes,
                                cbr_stream_t stream) {
  size_t need = 0;
  int st = check_forward_train(desc, x, w, gamma, beta, running_mean, running_var, momentum, eps, y,
                               relu_mask, z_saved, saved_mean, saved_inv_var, &need);
  if (st) return (cbr_status_t)st;
  if (!ws) return CBR_ERR_INVALID_ARG;
  if (!aligned(ws, 16)) return CBR_ERR_MISALIGNED;
  if (ws_bytes < need) return CBR_ERR_WORKSPACE;
  Shape s;
  check_desc(desc, &s);
  const FwdWs L = fwd_ws(s, z_saved == nullptr);
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev))) return (cbr_status_t)st;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  void* z = z_saved ? z_saved : wsb + L.z;
  Prof prof(cs);

  FpropArgs a{};
  a.g = make_geom(s);
  a.z = z;
  a.part = reinterpret_cast<float*>(wsb + L.part);
  a.ticket = reinterpret_cast<uint32_t*>(wsb);
  a.gamma = gamma;
  a.beta = beta;
  a.running_mean = running_mean;
  a.running_var = running_var;
  a.saved_mean = saved_mean;
  a.saved_inv_var = saved_inv_var;
  a.eq = reinterpret_cast<float*>(wsb + L.eq);
  a.momentum = momentum;
  a.eps = eps;
  a.m_count = s.m;
  a.err = dev->err;
  a.mode = kFpropStats;
  if (persistent) {
    if (is_first_layer(s) || s.stride != 1 || !aligned(y, 32) ||
        !fprop_apply_supported(a.g, (int)s.cin, (int)s.cout, dev->num_sms))
      return CBR_ERR_UNSUPPORTED;
    st = launch_fprop_apply(a, y, relu_mask, reinterpret_cast<uint32_t*>(wsb) + kReadyWord, (int)s.cin,
                            (int)s.cout, s.bf16, x, w, dev->num_sms, cs);
    if (st) return (cbr_status_t)st;
    prof.mark();
    return CBR_OK;
  }
  // The convolution writes its per-CTA partial moments and the apply pass merges and
  // finalizes them in its prologue (where the partials fit its shared memory); otherwise the
  // convolution's last CTA finalizes.
  int nparts = 0;
  a.defer = apply_merge_supported((int)s.cout, dev->num_sms) ? 1 : 0;
  a.parts_out = &nparts;
  st = run_fprop(a, s, x, w, dev->num_sms, cs);
  if (st) return (cbr_status_t)st;
  prof.mark();

  ApplyArgs ap{};
  ap.z = z;
  ap.y = y;
  ap.mask = reinterpret_cast<uint8_t*>(relu_mask);
  ap.eq = a.eq;
  ap.total = s.m * s.cout;
  ap.c = (int)s.cout;
  if (a.defer) {
    ap.part = a.part;
    ap.nparts = nparts;
    ap.gamma = gamma;
    ap.beta = beta;
    ap.running_mean = running_mean;
    ap.running_var = running_var;
    ap.saved_mean = saved_mean;
    ap.saved_inv_var = saved_inv_var;
    ap.momentum = momentum;
    ap.eps = eps;
    ap.inv_m = (float)(1.0 / (double)s.m);
    ap.unbias = s.m > 1 ? (float)((double)s.m / (double)(s.m - 1)) : 1.f;
    ap.err = dev->err;
  }
  st = launch_apply(ap, s.bf16, dev->num_sms, cs);
  if (st) return (cbr_status_t)st;
  prof.mark();
  return CBR_OK;
}

}  // namespace

extern "C" {

cbr_status_t cbr_forward_train(const cbr_desc_t* desc, const void* x, const void* w,
                               const float* gamma, const float* beta, float* running_mean,
                               float* running_var, float momentum, float eps, void* y,
                               uint32_t* relu_mask, void* z_saved, float* saved_mean,
                               float* saved_inv_var, void* ws, size_t ws_bytes,
                               cbr_stream_t stream) {
  return forward_train_impl(false, desc, x, w, gamma, beta, running_mean, running_var, momentum, eps, y, relu_mask,
                            z_saved, saved_mean, saved_inv_var, ws, ws_bytes, stream);
}

cbr_status_t cbr_forward_train_persistent(const cbr_desc_t* desc, const void* x, const void* w,
                                          const float* gamma, const float* beta, float* running_mean,
                                          float* running_var, float momentum, float eps, void* y,
                                          uint32_t* relu_mask, void* z_saved, float* saved_mean,
                                          float* saved_inv_var, void* ws, size_t ws_bytes,
                                          cbr_stream_t stream) {
  return forward_train_impl(true, desc, x, w, gamma, beta, running_mean, running_var, momentum, eps, y, relu_mask,
                            z_saved, saved_mean, saved_inv_var, ws, ws_bytes, stream);
}

cbr_status_t cbr_forward_train_stats(const cbr_desc_t* desc, const void* x, const void* w, void* z,
                                     float* moments, void* ws, size_t ws_bytes, cbr_stream_t stream) {
  Shape s;
  int st = check_desc(desc, &s);
  if (st) return (cbr_status_t)st;
  if (!x || !w || !z || !moments || !ws) return CBR_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(z, 16) || !aligned(ws, 16) || !aligned(moments, 4))
    return CBR_ERR_MISALIGNED;
  if ((st = check_supported(s))) return (cbr_status_t)st;
  const FwdWs L = fwd_ws(s, false);
  if (ws_bytes < L.total) return CBR_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev))) return (cbr_status_t)st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  Prof prof(cs);
  FpropArgs a{};
  a.g = make_geom(s);
  a.z = z;
  a.part = reinterpret_cast<float*>(wsb + L.part);
  a.ticket = reinterpret_cast<uint32_t*>(wsb);
  a.moments = moments;
  a.m_count = s.m;
  a.err = dev->err;
  a.mode = kFpropStats;
  st = run_fprop(a, s, x, w, dev->num_sms, cs);
  if (st) return (cbr_status_t)st;
  prof.mark();
  return CBR_OK;
}

cbr_status_t cbr_forward_train_finish(const cbr_desc_t* desc, const float* moments_all, int32_t world,
                                      const float* gamma, const float* beta, float* running_mean,
                                      float* running_var, float momentum, float eps, const void* z,
                                      void* y, uint32_t* relu_mask, float* saved_mean,
                                      float* saved_inv_var, void* ws, size_t ws_bytes,
                                      cbr_stream_t stream) {
  Shape s;
  int st = check_desc(desc, &s);
  if (st) return (cbr_status_t)st;
  if (!moments_all || world < 1 || world > 65536 || !gamma || !beta || !running_mean || !running_var || !z ||
      !y || !saved_mean || !saved_inv_var || !ws)
    return CBR_ERR_INVALID_ARG;
  if (!(momentum >= 0.f && momentum <= 1.f) || !(eps > 0.f) || !std::isfinite(eps)) return CBR_ERR_INVALID_ARG;
  if (!aligned(z, 16) || !aligned(y, 16) || !aligned(ws, 16) || (relu_mask && !aligned(relu_mask, 4)) ||
      !aligned(moments_all, 4) || !aligned(gamma, 4) || !aligned(beta, 4) || !aligned(running_mean, 4) ||
      !aligned(running_var, 4) || !aligned(saved_mean, 4) || !aligned(saved_inv_var, 4))
    return CBR_ERR_MISALIGNED;
  if ((st = check_supported(s))) return (cbr_status_t)st;
  const FwdWs L = fwd_ws(s, false);
  if (ws_bytes < L.total) return CBR_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev))) return (cbr_status_t)st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  Prof prof(cs);
  float* eq = reinterpret_cast<float*>(wsb + L.eq);
  st = launch_merge_finalize(moments_all, world, (int)s.cout, gamma, beta, running_mean, running_var, momentum, eps,
                             saved_mean, saved_inv_var, eq, cs);
  if (st) return (cbr_status_t)st;
  prof.mark();
  ApplyArgs ap{};
  ap.z = z;
  ap.y = y;
  ap.mask = reinterpret_cast<uint8_t*>(relu_mask);
  ap.eq = eq;
  ap.total = s.m * s.cout;
  ap.c = (int)s.cout;
  st = launch_apply(ap, s.bf16, dev->num_sms, cs);
  if (st) return (cbr_status_t)st;
  prof.mark();
  return CBR_OK;
}

}  // extern "C"

namespace cbr {
namespace {

// The three uses of the backward path: the whole backward; the split backward's first half
// (the masked reduction's raw sums, then stop); its second half (coefficients from sums
// reduced over all ranks, then the convolutions).
enum BwdMode { kBwdFull, kBwdSums, kBwdFinish };

int backward_run(BwdMode mode, const cbr_desc_t* desc, const void* dy, const void* x, const void* w,
                 const void* y_or_relu_mask, int32_t mask_kind, const void* z_saved, const float* gamma,
                 const float* saved_mean, const float* saved_inv_var, void* dx, float* dw, float* dgamma,
                 float* dbeta, void* ws, size_t ws_bytes, cbr_stream_t stream, float* sums_out,
                 const float* sums_all, long long m_total) {
  Shape s;
  int st = check_desc(desc, &s);
  if (st) return (cbr_status_t)st;
  if (mode == kBwdSums) {
    // only the reduction runs: it reads dy, the mask and z against the mean
    if (!dy || !y_or_relu_mask || !z_saved || !saved_mean || !sums_out || !ws) return CBR_ERR_INVALID_ARG;
    // x, W, gamma, inv_std and the gradient outputs are not touched; aliases keep the shared
    // checks below simple (the sums need only 4-byte alignment)
    x = w = dy;
    gamma = saved_inv_var = dgamma = dbeta = dw = sums_out;
    dx = nullptr;
  } else if (!dy || !x || !w || !y_or_relu_mask || !gamma || !saved_mean || !saved_inv_var || !dw ||
             !dgamma || !dbeta || !ws) {
    return CBR_ERR_INVALID_ARG;
  }
  if (mode == kBwdFinish && (!sums_all || m_total < 2)) return CBR_ERR_INVALID_ARG;
  if (mask_kind != CBR_MASK_BITS && mask_kind != CBR_MASK_FROM_Y && mask_kind != CBR_MASK_BYTES)
    return CBR_ERR_INVALID_ARG;
  if (dx && overlaps(dx, act_bytes(s.n, s.h, s.w, s.cin, s.elt), x,
                     act_bytes(s.n, s.h, s.w, s.cin, s.elt)))
    return CBR_ERR_INVALID_ARG;
  if (!aligned(dy, 16) || !aligned(x, 16) || !aligned(w, 16) || !aligned(ws, 16) ||
      (dx && !aligned(dx, 16)) || (z_saved && !aligned(z_saved, 16)) ||
      !aligned(y_or_relu_mask, mask_kind == CBR_MASK_BITS ? 4 : 16) || (mode != kBwdSums && !aligned(dw, 16)) ||
      !aligned(gamma, 4) || !aligned(saved_mean, 4) || !aligned(saved_inv_var, 4) ||
      !aligned(dgamma, 4) || !aligned(dbeta, 4))
    return CBR_ERR_MISALIGNED;
  if ((st = check_supported(s))) return (cbr_status_t)st;
  // dgrad runs as a stride-1 conv with padding R-1-pad on both axes
  if (dx && (s.r != s.s || s.pad > s.r - 1)) return CBR_ERR_UNSUPPORTED;
  // The first layer has no dgrad (CBR page, section 5.3): dx must be NULL there.
  if (is_first_layer(s) && dx) return CBR_ERR_UNSUPPORTED;
  const BwdWs L = bwd_ws(s, z_saved == nullptr);
  if (ws_bytes < L.total) return CBR_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev))) return (cbr_status_t)st;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  Prof prof(cs);
  const void* z = z_saved;
  if (!z) {
    // recompute z = conv(x, W) (no statistics)
    FpropArgs a{};
    a.g = make_geom(s);
    a.z = wsb + L.z;
    a.m_count = s.m;
    a.err = dev->err;
    a.mode = kFpropPlain;
    st = run_fprop(a, s, x, w, dev->num_sms, cs);
    if (st) return (cbr_status_t)st;
    prof.mark();
    z = wsb + L.z;
  }
  const uint8_t* mask = mask_kind == CBR_MASK_BITS ? static_cast<const uint8_t*>(y_or_relu_mask) : nullptr;
  const void* yv = mask_kind == CBR_MASK_FROM_Y ? y_or_relu_mask : nullptr;
  if (mask_kind == CBR_MASK_BYTES) {
    // a byte-per-element mask is packed into the workspace once; the kernels read bits
    uint32_t* mb = reinterpret_cast<uint32_t*>(wsb + L.mbits);
    st = launch_mask_bytes_to_bits(static_cast<const uint8_t*>(y_or_relu_mask), mb, s.m * s.cout, dev->num_sms, cs);
    if (st) return (cbr_status_t)st;
    prof.mark();
    mask = reinterpret_cast<const uint8_t*>(mb);
  }
  float* coef = reinterpret_cast<float*>(wsb + L.coef);

  if (mode == kBwdFinish) {
    // sums reduced over all ranks: dgamma, dbeta and the coefficients over the global batch
    st = launch_bwd_coef(sums_all, (int)s.cout, m_total, gamma, saved_mean, saved_inv_var, dgamma, dbeta, coef, cs);
    if (st) return (cbr_status_t)st;
    prof.mark();
  } else {
    BwdReduceArgs b{};
    b.dy = dy;
    b.z = z;
    b.y = yv;
    b.mask = mask;
    b.gamma = gamma;
    b.mean = saved_mean;
    b.inv_std = saved_inv_var;
    b.dgamma = dgamma;
    b.dbeta = dbeta;
    b.coef = coef;
    b.sums_out = mode == kBwdSums ? sums_out : nullptr;
    b.part = reinterpret_cast<float*>(wsb + L.part);
    b.ticket = reinterpret_cast<uint32_t*>(wsb) + 1;
    b.m_count = s.m;
    b.c = (int)s.cout;
    b.err = dev->err;
    st = launch_bwd_reduce(b, s.bf16, dev->num_sms, cs);
    if (st) return (cbr_status_t)st;
    prof.mark();
    if (mode == kBwdSums) return CBR_OK;
  }

  if (use_fused_bwd(s)) {
    // dz = a*(dy*mask) - d*z + e evaluated once per tile on chip, feeding both convolutions
    BwdFusedArgs fa{};
    fa.g = make_geom(s);
    fa.dy = dy;
    fa.z = z;
    fa.y = yv;
    fa.mask = mask;
    fa.coef = coef;
    fa.dx = dx;
    fa.part = reinterpret_cast<float*>(wsb + L.wpart);
    fa.dw = dw;
    fa.err = dev->err;
    st = launch_bwd_fused(fa, (int)s.cin, (int)s.cout, s.bf16, x, w, dev->num_sms, cs,
                          [](void* p) { static_cast<Prof*>(p)->mark(); }, &prof);
    if (st) return (cbr_status_t)st;
    prof.mark();
    return CBR_OK;
  }

  // Other layers: dz = a*(dy*mask) - d*z + e is materialised once and read by TMA in both
  // convolutions.
  if (!dz_materialisable(s)) return CBR_ERR_UNSUPPORTED;
  void* dz_buf = wsb + L.dz;
  {
    DzArgs za{};
    za.dy = dy;
    za.z = z;
    za.y = yv;
    za.mask = mask;
    za.coef = coef;
    za.dz = dz_buf;
    za.total = s.m * s.cout;
    za.c = (int)s.cout;
    za.q = (int)s.q;
    za.pitch = (int)dz_pitch(s);
    st = launch_dz(za, s.bf16, dev->num_sms, cs);
    if (st) return (cbr_status_t)st;
    prof.mark();
  }

  if (is_first_layer(s)) {
    // first layer: the im2col wgrad over the materialised dz; no dgrad (CBR page, section 5.3)
    st = launch_first_wgrad(make_geom(s), (int)s.stride, (int)s.cout, s.bf16, x, dz_buf,
                            reinterpret_cast<float*>(wsb + L.wpart), dw, dev->err, dev->num_sms, cs,
                            [](void* p) { static_cast<Prof*>(p)->mark(); }, &prof);
    if (st) return (cbr_status_t)st;
    prof.mark();
    return CBR_OK;
  }

  // WGrad first, then DGrad (CBR page, section 5.2 orders DGrad after WGrad because its dX
  // overwrote X there; here dx may not alias x, so the order is only kept for familiarity).
  if (!wgrad_dz_tma_fits(make_geom(s), (int)s.cout)) return CBR_ERR_UNSUPPORTED;
  WgradArgs wa{};
  wa.dz_full = dz_buf;
  wa.g = make_geom(s);
  wa.part = reinterpret_cast<float*>(wsb + L.wpart);
  wa.dw = dw;
  wa.err = dev->err;
  st = launch_wgrad(wa, (int)s.cin, (int)s.cout, s.bf16, x, dev->num_sms, cs,
                    [](void* p) { static_cast<Prof*>(p)->mark(); }, &prof);
  if (st) return (cbr_status_t)st;
  prof.mark();

  if (dx) {
    DgradArgs da{};
    // dgrad = stride-1 conv of dz (P x Q, cout channels) with the flipped filter, pad R-1-pad
    da.g.n_img = (int)s.n;
    da.g.h = (int)s.p;
    da.g.w = (int)s.q;
    da.g.r = (int)s.r;
    da.g.s = (int)s.s;
    da.g.pad = (int)(s.r - 1 - s.pad);
    da.dx = dx;
    da.dz_full = dz_buf;
    da.dz_pitch = (int)dz_pitch(s);
    da.err = dev->err;
    st = launch_dgrad(da, (int)s.cin, (int)s.cout, s.bf16, w, dev->num_sms, cs);
    if (st) return (cbr_status_t)st;
    prof.mark();
  }
  return CBR_OK;
}

}  // namespace
}  // namespace cbr

extern "C" {

cbr_status_t cbr_backward(const cbr_desc_t* desc, const void* dy, const void* x, const void* w,
                          const void* y_or_relu_mask, int32_t mask_kind, const void* z_saved,
                          const float* gamma, const float* saved_mean,
                          const float* saved_inv_var, void* dx, float* dw, float* dgamma,
                          float* dbeta, void* ws, size_t ws_bytes, cbr_stream_t stream) {
  return (cbr_status_t)backward_run(kBwdFull, desc, dy, x, w, y_or_relu_mask, mask_kind, z_saved, gamma,
                                    saved_mean, saved_inv_var, dx, dw, dgamma, dbeta, ws, ws_bytes, stream,
                                    nullptr, nullptr, 0);
}

cbr_status_t cbr_backward_sums(const cbr_desc_t* desc, const void* dy, const void* y_or_relu_mask,
                               int32_t mask_kind, const void* z_saved, const float* saved_mean,
                               float* sums, void* ws, size_t ws_bytes, cbr_stream_t stream) {
  return (cbr_status_t)backward_run(kBwdSums, desc, dy, nullptr, nullptr, y_or_relu_mask, mask_kind, z_saved,
                                    nullptr, saved_mean, nullptr, nullptr, nullptr, nullptr, nullptr, ws,
                                    ws_bytes, stream, sums, nullptr, 0);
}

cbr_status_t cbr_backward_finish(const cbr_desc_t* desc, const float* sums_all, int64_t m_total,
                                 const void* dy, const void* x, const void* w,
                                 const void* y_or_relu_mask, int32_t mask_kind, const void* z_saved,
                                 const float* gamma, const float* saved_mean,
                                 const float* saved_inv_var, void* dx, float* dw, float* dgamma,
                                 float* dbeta, void* ws, size_t ws_bytes, cbr_stream_t stream) {
  return (cbr_status_t)backward_run(kBwdFinish, desc, dy, x, w, y_or_relu_mask, mask_kind, z_saved, gamma,
                                    saved_mean, saved_inv_var, dx, dw, dgamma, dbeta, ws, ws_bytes, stream,
                                    nullptr, sums_all, m_total);
}

cbr_status_t cbr_fold_bn(const cbr_desc_t* desc, const void* w, const float* conv_bias,
                         const float* gamma, const float* beta, const float* running_mean,
                         const float* running_var, float eps, void* w_fold, float* b_fold,
                         cbr_stream_t stream) {
  Shape s;
  int st = check_desc(desc, &s);
  if (st) return (cbr_status_t)st;
  if (!w || !gamma || !beta || !running_mean || !running_var || !w_fold || !b_fold)
    return CBR_ERR_INVALID_ARG;
  if (!(eps > 0.f) || !std::isfinite(eps)) return CBR_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(w_fold, 16) || !aligned(gamma, 4) || !aligned(beta, 4) ||
      !aligned(running_mean, 4) || !aligned(running_var, 4) || !aligned(b_fold, 4) ||
      (conv_bias && !aligned(conv_bias, 4)))
    return CBR_ERR_MISALIGNED;
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev))) return (cbr_status_t)st;
  return (cbr_status_t)launch_fold(w, conv_bias, gamma, beta, running_mean, running_var, eps,
                                   w_fold, b_fold, (int)s.cout, (int)(s.r * s.s * s.cin), s.bf16,
                                   reinterpret_cast<cudaStream_t>(stream));
}

cbr_status_t cbr_forward_infer(const cbr_desc_t* desc, const void* x, const void* w_fold,
                               const float* b_fold, void* y, cbr_stream_t stream) {
  Shape s;
  int st = check_desc(desc, &s);
  if (st) return (cbr_status_t)st;
  if (!x || !w_fold || !b_fold || !y) return CBR_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_fold, 16) || !aligned(y, 16) || !aligned(b_fold, 4))
    return CBR_ERR_MISALIGNED;
  if ((st = check_supported(s))) return (cbr_status_t)st;
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev))) return (cbr_status_t)st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  Prof prof(cs);
  FpropArgs a{};
  a.g = make_geom(s);
  a.z = y;
  a.bias = b_fold;
  a.m_count = s.m;
  a.err = dev->err;
  a.mode = kFpropBiasRelu;
  st = run_fprop(a, s, x, w_fold, dev->num_sms, cs);
  if (st) return (cbr_status_t)st;
  prof.mark();
  return CBR_OK;
}

cbr_status_t cbr_mask_bits_to_bytes(const uint32_t* bits, uint8_t* bytes, int64_t count,
                                    cbr_stream_t stream) {
  if (count < 0 || (count > 0 && (!bits || !bytes))) return CBR_ERR_INVALID_ARG;
  if (count == 0) return CBR_OK;
  if (!aligned(bits, 4) || !aligned(bytes, 16)) return CBR_ERR_MISALIGNED;
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st) return (cbr_status_t)st;
  return (cbr_status_t)launch_mask_bits_to_bytes(bits, bytes, count, dev->num_sms,
                                                 reinterpret_cast<cudaStream_t>(stream));
}

cbr_status_t cbr_mask_bytes_to_bits(const uint8_t* bytes, uint32_t* bits, int64_t count,
                                    cbr_stream_t stream) {
  if (count < 0 || (count > 0 && (!bits || !bytes))) return CBR_ERR_INVALID_ARG;
  if (count == 0) return CBR_OK;
  if (!aligned(bits, 4) || !aligned(bytes, 16)) return CBR_ERR_MISALIGNED;
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st) return (cbr_status_t)st;
  return (cbr_status_t)launch_mask_bytes_to_bits(bytes, bits, count, dev->num_sms,
                                                 reinterpret_cast<cudaStream_t>(stream));
}

cbr_status_t cbr_forward_infer_bn(const cbr_desc_t* desc, const void* x, const void* w,
                                  const float* conv_bias, const float* gamma, const float* beta,
                                  const float* running_mean, const float* running_var, float eps,
                                  void* y, cbr_stream_t stream) {
  Shape s;
  int st = check_desc(desc, &s);
  if (st) return (cbr_status_t)st;
  if (!x || !w || !gamma || !beta || !running_mean || !running_var || !y) return CBR_ERR_INVALID_ARG;
  if (!(eps > 0.f) || !std::isfinite(eps)) return CBR_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(gamma, 4) || !aligned(beta, 4) ||
      !aligned(running_mean, 4) || !aligned(running_var, 4) || (conv_bias && !aligned(conv_bias, 4)))
    return CBR_ERR_MISALIGNED;
  if ((st = check_supported(s))) return (cbr_status_t)st;
  // the 3-channel first layer has its own kernels, which take the folded form only
  if (is_first_layer(s)) return CBR_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev))) return (cbr_status_t)st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  Prof prof(cs);
  FpropArgs a{};
  a.g = make_geom(s);
  a.z = y;
  a.eps = eps;
  a.bn_gamma = gamma;
  a.bn_beta = beta;
  a.bn_mean = running_mean;
  a.bn_var = running_var;
  a.conv_bias = conv_bias;
  a.m_count = s.m;
  a.err = dev->err;
  st = launch_fprop_bn(a, (int)s.cin, (int)s.cout, s.bf16, x, w, dev->num_sms, cs);
  if (st) return (cbr_status_t)st;
  prof.mark();
  return CBR_OK;
}

cbr_status_t cbr_stream_status(cbr_stream_t stream) {
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st) return (cbr_status_t)st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return CBR_ERR_CUDA;
  }
  uint32_t word = 0;
  if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word)) != cudaSuccess) return CBR_ERR_CUDA;
  if (word) {
    const uint32_t zero = 0;
    cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    return CBR_ERR_TIMEOUT;
  }
  return CBR_OK;
}

cbr_status_t cbr_selftest_bounded_wait(int32_t limit_us, cbr_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return CBR_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st) return (cbr_status_t)st;
  st = launch_selftest_wait(dev->err, (uint64_t)limit_us * 1000ull, reinterpret_cast<cudaStream_t>(stream));
  return (cbr_status_t)st;
}

cbr_status_t cbr_profile_next_call(void* const* events, int32_t count) {
  if (events && count <= 0) return CBR_ERR_INVALID_ARG;
  t_prof_events = events;
  t_prof_count = events ? count : 0;
  return CBR_OK;
}

int32_t cbr_profile_last_count(void) { return t_prof_used; }

}  // extern "C"
