// ga.cu -- the C ABI of libga (declared in include/ga.h): argument validation, TMA tensor
// maps, kernel selection and launch.  Every entry point validates on the host before any
// CUDA call and returns a ga_status; nothing here allocates device memory.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <utility>
#include <atomic>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/ga.h"
#include "attend_simt.cuh"
#include "blocks.cuh"
#include "common.cuh"
#include "decode.cuh"
#include "dsa.cuh"
#include "mla.cuh"
#include "prefill_wide.cuh"
#include "ring.cuh"
#include "select.cuh"

namespace ga {

namespace {

uint64_t g_timeout_ns = 2000000000ull;
int g_test_drop_chunk = -1;    // test only: ring chunk the prefill producer of CTA 0 skips
std::atomic<unsigned> g_wide_epoch{0};   // launch counter: each prefill launch's item-counter slot

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda) --------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D bf16 map over a [planes, rows, cols] row-major tensor, boxes of box_rows x 64 columns
// with the 128-byte swizzle; out-of-range rows read as zero.
bool make_map_bf16(CUtensorMap* map, const void* base, int cols, long long rows, long long planes,
                   int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * 2 * (cuuint64_t)rows};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp32 map over a [planes, rows, cols] row-major tensor, boxes of box_rows x 32 columns
// (128 bytes) with the 128-byte swizzle; out-of-range rows read as zero.
bool make_map_f32(CUtensorMap* map, const void* base, int cols, long long rows, long long planes,
                  int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 4, (cuuint64_t)cols * 4 * (cuuint64_t)rows};
  cuuint32_t box[3] = {32, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches kernel<<<grid, block, smem, stream>>>(args...) with programmatic stream
// serialization: it may start while the previous kernel on the stream finishes, and waits for it
// (griddep_wait) only where it reads that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename K>
int set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess
             ? GA_OK
             : GA_ERR_CUDA;
}

// Kernels that move registers between warpgroups with setmaxnreg: the increase waits until the
// registers exist, so the CTA must have been launched with at least `need` registers in all.
template <typename K>
int set_smem_split(K kernel, int bytes, int threads, int need) {
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, kernel) != cudaSuccess) return GA_ERR_CUDA;
  if (attr.numRegs * threads < need) return GA_ERR_UNSUPPORTED;
  return set_smem(kernel, bytes);
}

int launch_status() { return cudaGetLastError() == cudaSuccess ? GA_OK : GA_ERR_CUDA; }

// ---- split-K decode geometry (shared by ga_workspace_size and ga_attend) -----------------
bool decode_eligible(int n_heads, int n_kv, int d, int Tq, ga_dtype dtype, const void* block_mask) {
  const int g = n_heads / n_kv;
  return dtype == GA_BF16 && block_mask == nullptr && (d == 64 || d == 128 || d == 256) && (long long)g * Tq <= 16;
}

int decode_chunk_len(int batch, int n_kv, int Tk_max) {
  const long long want = (long long)Tk_max * batch * n_kv / (148LL * 8);
  long long c = (want + 63) / 64 * 64;
  if (c < 512) c = 512;
  if (c > 4096) c = 4096;
  return (int)c;
}

int tc_eligible(int d, ga_dtype dtype, const void* q, const void* k, const void* v, const void* out,
                const void* block_mask, int q_block, int k_block) {
  if (dtype != GA_BF16 || !(d == 128 || d == 256)) return 0;
  if (block_mask && (q_block % 128 != 0 || k_block % 64 != 0)) return 0;
  return aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out);
}

}  // namespace

// ---- self-test kernel for the bounded wait ------------------------------------------------
__global__ void selftest_wait_kernel(const volatile int* flag, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer();
  while (*flag == 0) {
    if (globaltimer() - t0 > timeout_ns) {
      record_status(GA_ERR_DEVICE_TIMEOUT);
      return;
    }
    __nanosleep(1000);
  }
}

__device__ int g_never_set_flag = 0;

// Scratch of ga_attend_decode_static: the split-K partial rows and their (max, sum) pairs.
// Every device that loads the library holds it until the process exits.
static __device__ __align__(256) unsigned char g_decode_static_scratch[GA_DECODE_STATIC_SCRATCH_BYTES];

namespace {

// ---- once per device: kernel attributes and properties -----------------------------------
// cudaFuncSetAttribute applies to the device current when it is called, so every device a
// process launches on gets its own set-up, the first time an entry point runs there.  Each
// kernel family keeps its own status (a family whose register budget does not fit is
// refused on its own); the record never changes once filled.
constexpr int kMaxDevices = 128;

struct DeviceKernels {
  int prefill128, prefill256;   // prefill_wide_kernel at d = 128 / 256 (every epilogue mode)
  int decode;                   // decode_splitk_kernel, plain and gathered
  int select;                   // select_blocks_kernel
  int mla;                      // mla_decode_kernel
  int topk, topk_unstaged;      // topk_select_kernel with / without the row staged in shared memory
  int n_sm;                     // streaming multiprocessors
  long long l2_bytes;           // L2 cache size
};

std::mutex g_dev_mu;
bool g_dev_ready[kMaxDevices] = {};
DeviceKernels g_dev[kMaxDevices];

int first_error(std::initializer_list<int> sts) {
  for (int s : sts)
    if (s != GA_OK) return s;
  return GA_OK;
}

// The set-up record of the device current in the calling thread (null when that device cannot
// be queried).
const DeviceKernels* device_kernels() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!g_dev_ready[dev]) {
    DeviceKernels& d = g_dev[dev];
    {
      using C = WideCfg<128>;
      constexpr int need = 256 * C::SOFTMAX_REGS + 128 * C::OTHER_REGS;
      d.prefill128 = first_error({set_smem_split(prefill_wide_kernel<128, false>, C::SMEM_BYTES, C::THREADS, need),
                                  set_smem_split(prefill_wide_kernel<128, true>, C::SMEM_BYTES, C::THREADS, need),
                                  set_smem_split(prefill_wide_kernel<128, false, 1>, C::SMEM_BYTES, C::THREADS, need),
                                  set_smem_split(prefill_wide_kernel<128, false, 2>, C::SMEM_BYTES, C::THREADS, need)});
    }
    {
      using C = WideCfg<256>;
      d.prefill256 = first_error({set_smem(prefill_wide_kernel<256, false>, C::SMEM_BYTES),
                                  set_smem(prefill_wide_kernel<256, true>, C::SMEM_BYTES),
                                  set_smem(prefill_wide_kernel<256, false, 1>, C::SMEM_BYTES),
                                  set_smem(prefill_wide_kernel<256, false, 2>, C::SMEM_BYTES)});
    }
    d.decode = first_error({set_smem(decode_splitk_kernel<256, false>, DecodeCfg<256>::SMEM_BYTES),
                            set_smem(decode_splitk_kernel<128, false>, DecodeCfg<128>::SMEM_BYTES),
                            set_smem(decode_splitk_kernel<64, false>, DecodeCfg<64>::SMEM_BYTES),
                            set_smem(decode_splitk_kernel<256, true>, DecodeCfg<256>::GATHER_SMEM_BYTES),
                            set_smem(decode_splitk_kernel<128, true>, DecodeCfg<128>::GATHER_SMEM_BYTES),
                            set_smem(decode_splitk_kernel<64, true>, DecodeCfg<64>::GATHER_SMEM_BYTES)});
    d.select = first_error({set_smem(select_rescue_kernel, 16384 * 8), set_smem(select_score_kernel, kScSmem)});
    d.mla = set_smem(mla_decode_kernel, MlaCfg::SMEM_BYTES);
    if (d.mla == GA_OK) d.mla = set_smem(mla_expand_kernel, MlaCfg::EX_SMEM);
    d.topk = set_smem(topk_select_kernel<true>, kTopkFixedSmem + kTopkStageMax * 4);
    d.topk_unstaged = set_smem(topk_select_kernel<false>, kTopkFixedSmem);
    int n_sm = 0;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm < 1) n_sm = 148;
    d.n_sm = n_sm;
    int l2 = 0;
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 < 1) l2 = 126 << 20;
    d.l2_bytes = l2;
    g_dev_ready[dev] = true;
  }
  return &g_dev[dev];
}

// Device address of g_decode_static_scratch on the current device.  Host code must not use
// the symbol itself as a pointer (on the host it names a stand-in, not device memory), so
// the address is looked up once per device, with that device current, and cached.
std::mutex g_static_mu;
void* g_static_scratch_addr[kMaxDevices] = {};

int static_scratch_setup(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_static_scratch) != cudaSuccess || p == nullptr)
      return GA_ERR_CUDA;
    g_static_scratch_addr[dev] = p;
  }
  *addr = g_static_scratch_addr[dev];
  return GA_OK;
}

// Launches the split-K decode (d in {64, 128, 256}) and, for more than one chunk, the combine.
// The caller has validated the shape and placed the partial-result workspace.
template <int D, bool GATHER>
int launch_decode_d(const CUtensorMap& tk, const CUtensorMap& tv, const __nv_bfloat16* qb,
                    __nv_bfloat16* ob, float* lse, float* ws_o, float* ws_ml, const DecodeShape& ds,
                    cudaStream_t stream) {
  constexpr int smem = GATHER ? DecodeCfg<D>::GATHER_SMEM_BYTES : DecodeCfg<D>::SMEM_BYTES;
  const DeviceKernels* dk = device_kernels();
  if (!dk) return GA_ERR_CUDA;
  if (dk->decode != GA_OK) return dk->decode;
  const dim3 grid(ds.n_chunks, ds.a.n_kv, ds.a.batch);
  if (GATHER) {
    // a programmatic dependent of the previous kernel (the top-k select's index lists)
    if (launch_pdl(decode_splitk_kernel<D, GATHER>, grid, dim3(DecodeCfg<D>::THREADS), smem, stream, tk, tv, qb, ob,
                   lse, ws_o, ws_ml, ds) != cudaSuccess)
      return GA_ERR_CUDA;
  } else {
    decode_splitk_kernel<D, GATHER><<<grid, DecodeCfg<D>::THREADS, smem, stream>>>(
        tk, tv, qb, ob, lse, ws_o, ws_ml, ds);
  }
  const int st = launch_status();
  if (st != GA_OK || ds.n_chunks == 1) return st;
  if (launch_pdl(decode_combine_kernel<D>, dim3(ds.a.Tq, ds.a.n_heads, ds.a.batch), dim3(D), 0, stream, ws_o,
                 ws_ml, ob, lse, ds) != cudaSuccess)
    return GA_ERR_CUDA;
  return launch_status();
}

int launch_decode(int d, const CUtensorMap& tk, const CUtensorMap& tv, const __nv_bfloat16* qb,
                  __nv_bfloat16* ob, float* lse, float* ws_o, float* ws_ml, const DecodeShape& ds,
                  cudaStream_t stream, bool gather = false) {
  if (gather) {
    if (d == 256) return launch_decode_d<256, true>(tk, tv, qb, ob, lse, ws_o, ws_ml, ds, stream);
    if (d == 128) return launch_decode_d<128, true>(tk, tv, qb, ob, lse, ws_o, ws_ml, ds, stream);
    return launch_decode_d<64, true>(tk, tv, qb, ob, lse, ws_o, ws_ml, ds, stream);
  }
  if (d == 256) return launch_decode_d<256, false>(tk, tv, qb, ob, lse, ws_o, ws_ml, ds, stream);
  if (d == 128) return launch_decode_d<128, false>(tk, tv, qb, ob, lse, ws_o, ws_ml, ds, stream);
  return launch_decode_d<64, false>(tk, tv, qb, ob, lse, ws_o, ws_ml, ds, stream);
}

// The tensor-core prefill (bf16, d = 128 or 256): tensor maps, then prefill_wide_kernel with or
// without block-mask unit lists.  The caller has validated the shape.
int launch_prefill_tc(const void* q, const void* k, const void* v, __nv_bfloat16* ob, float* lse,
                      const AttnShape& sh_in, bool masked, WideEpi epi, cudaStream_t stream) {
  AttnShape sh = sh_in;
  const int d = sh.d, Tq = sh.Tq, Tk_max = sh.Tk_max;
  // 64-column SW128 boxes: Q 128 rows; K 128 keys and 64 keys; V 16384/d keys and 64 keys
  const long long kvz = (long long)sh.batch * sh.n_kv;
  const int vk = 16384 / d;
  CUtensorMap tq, tk, tv, tk64, tv64;
  if (!make_map_bf16(&tq, q, d, Tq, (long long)sh.batch * sh.n_heads, 128) ||
      !make_map_bf16(&tk, k, d, Tk_max, kvz, 128) || !make_map_bf16(&tv, v, d, Tk_max, kvz, vk) ||
      !make_map_bf16(&tk64, k, d, Tk_max, kvz, 64) || !make_map_bf16(&tv64, v, d, Tk_max, kvz, 64))
    return GA_ERR_CUDA;
  const long long n_items = wide_items(sh);
  if (n_items > 0x7fffffffLL) return GA_ERR_UNSUPPORTED;
  const DeviceKernels* dk = device_kernels();
  if (!dk) return GA_ERR_CUDA;
  // persistent: one CTA per SM (or per item when there are fewer items)
  const unsigned n_cta = (unsigned)(n_items < dk->n_sm ? n_items : dk->n_sm);
  // Item order: when the keys and values of the launch do not fit in L2 and every query tile
  // reads all of its sequence's keys (no window), neighbouring query tiles of a kv head are
  // claimed together (blocks of 4), so that their reads of the same keys meet in L2; otherwise
  // the plain order, whose concurrent items already share their keys in L2.
  const double kv_bytes = 4.0 * sh.batch * sh.n_kv * (double)Tk_max * d;
  const int QB = (sh.window == 0 && kv_bytes > (double)dk->l2_bytes &&
                  4LL * sh.n_heads * sh.batch <= 0x7fffffffLL) ? 4 : 1;
  const int n_qt = (Tq + 127) / 128, g = sh.n_heads / sh.n_kv;
  sh.item_qt_block = QB;
  sh.fd_hb.init((uint32_t)(sh.n_heads * sh.batch));
  sh.fd_h.init((uint32_t)sh.n_heads);
  sh.fd_g.init((uint32_t)g);
  sh.fd_nkv.init((uint32_t)sh.n_kv);
  sh.fd_pb.init((uint32_t)(QB * sh.n_heads * sh.batch));
  sh.fd_cg.init((uint32_t)(QB * g));
  sh.fd_cgl.init((uint32_t)((n_qt - QB * ((n_qt - 1) / QB)) * g));   // query tiles of the last block x g
  const int epoch = (int)(g_wide_epoch.fetch_add(1u) % (unsigned)kWideEpochs);
  if (d == 128) {
    using C = WideCfg<128>;
    static_assert(C::VK == 128, "V map box");
    if (dk->prefill128 != GA_OK) return dk->prefill128;
    auto kern = epi.mode == 1 ? prefill_wide_kernel<128, false, 1>
              : epi.mode == 2 ? prefill_wide_kernel<128, false, 2>
              : masked        ? prefill_wide_kernel<128, true>
                              : prefill_wide_kernel<128, false>;
    kern<<<n_cta, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, tk64, tv64, ob, lse, sh, epi, epoch, g_test_drop_chunk);
  } else {
    using C = WideCfg<256>;
    static_assert(C::VK == 64, "V map box");
    if (dk->prefill256 != GA_OK) return dk->prefill256;
    auto kern = epi.mode == 1 ? prefill_wide_kernel<256, false, 1>
              : epi.mode == 2 ? prefill_wide_kernel<256, false, 2>
              : masked        ? prefill_wide_kernel<256, true>
                              : prefill_wide_kernel<256, false>;
    kern<<<n_cta, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, tk64, tv64, ob, lse, sh, epi, epoch, g_test_drop_chunk);
  }
  return launch_status();
}

}  // namespace

}  // namespace ga

using namespace ga;

extern "C" {

int ga_version(void) { return 100; }

const char* ga_status_string(int status) {
  switch (status) {
    case GA_OK: return "GA_OK";
    case GA_ERR_INVALID_ARG: return "GA_ERR_INVALID_ARG: invalid size, pointer, alignment or combination";
    case GA_ERR_UNSUPPORTED: return "GA_ERR_UNSUPPORTED: valid but not implemented by the kernels";
    case GA_ERR_CUDA: return "GA_ERR_CUDA: a CUDA call failed";
    case GA_ERR_DEVICE_TIMEOUT: return "GA_ERR_DEVICE_TIMEOUT: a device-side wait ran past its limit";
    case GA_ERR_WORKSPACE: return "GA_ERR_WORKSPACE: workspace missing or too small";
    case GA_ERR_SCRATCH_LIMIT:
      return "GA_ERR_SCRATCH_LIMIT: the shape needs more scratch than the library's static array "
             "(GA_DECODE_STATIC_SCRATCH_BYTES) holds";
    default: return "unknown ga_status";
  }
}

void ga_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns = ns < 100000ull ? 100000ull : ns; }

int ga_read_device_status(ga_stream_t stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GA_ERR_CUDA;
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return GA_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return GA_ERR_CUDA;
  return v;
}

void ga_selftest_drop_prefill_chunk(int chunk) { g_test_drop_chunk = chunk < 0 ? -1 : chunk; }

int ga_debug_violation(uint64_t* first, ga_stream_t stream) {
#ifdef GA_DEBUG
  if (!first) return GA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GA_ERR_CUDA;
  unsigned long long v = 0ull, zero = 0ull;
  if (cudaMemcpyFromSymbol(&v, g_debug_violation, sizeof(v)) != cudaSuccess) return GA_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_debug_violation, &zero, sizeof(zero)) != cudaSuccess) return GA_ERR_CUDA;
  *first = v;
  return GA_OK;
#else
  (void)first;
  (void)stream;
  return GA_ERR_UNSUPPORTED;
#endif
}

int ga_selftest_wait_timeout(uint64_t timeout_ns, ga_stream_t stream) {
  int* flag = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&flag), g_never_set_flag) != cudaSuccess)
    return GA_ERR_CUDA;
  selftest_wait_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(flag, timeout_ns);
  return launch_status();
}

size_t ga_workspace_size(int batch, int n_heads, int n_kv, int d, int Tq, int Tk_max, ga_dtype dtype) {
  if (batch < 1 || n_heads < 1 || n_kv < 1 || n_heads % n_kv != 0 || d < 1 || d > 256 || Tq < 1 ||
      Tk_max < Tq)
    return SIZE_MAX;
  if (!decode_eligible(n_heads, n_kv, d, Tq, dtype, nullptr)) return 0;
  const int chunk = decode_chunk_len(batch, n_kv, Tk_max);
  const int n_chunks = (Tk_max + chunk - 1) / chunk;
  if (n_chunks <= 1) return 0;
  return (size_t)batch * n_heads * Tq * n_chunks * (size_t)(d + 2) * sizeof(float);
}

int ga_attend(const void* q, const void* k, const void* v, void* out, int batch, int n_heads,
              int n_kv, int d, int Tq, int Tk_max, const int32_t* k_lens, int causal, int window,
              const float* sink, const uint8_t* block_mask, int q_block, int k_block, float* lse,
              ga_dtype dtype, void* workspace, size_t workspace_bytes, ga_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (!q || !k || !v || !out) return GA_ERR_INVALID_ARG;
  if (dtype != GA_F32 && dtype != GA_BF16) return GA_ERR_INVALID_ARG;
  if (batch < 1 || n_heads < 1 || n_kv < 1 || n_kv > n_heads || n_heads % n_kv != 0)
    return GA_ERR_INVALID_ARG;
  if (d < 1 || d > 256 || Tq < 1 || Tk_max < Tq) return GA_ERR_INVALID_ARG;
  if ((causal != 0 && causal != 1) || window < 0 || (window > 0 && !causal)) return GA_ERR_INVALID_ARG;
  if (block_mask && (q_block < 1 || k_block < 1)) return GA_ERR_INVALID_ARG;
  if (batch > 65535 || n_heads > 65535) return GA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (lse && !aligned16(lse)) || (sink && !aligned16(sink)) || (k_lens && !aligned16(k_lens)))
    return GA_ERR_INVALID_ARG;

  AttnShape sh{};
  sh.batch = batch; sh.n_heads = n_heads; sh.n_kv = n_kv; sh.d = d; sh.Tq = Tq; sh.Tk_max = Tk_max;
  sh.k_lens = k_lens; sh.causal = causal; sh.window = window; sh.sink = sink;
  sh.block_mask = block_mask;
  sh.q_block = block_mask ? q_block : 1;
  sh.k_block = block_mask ? k_block : 1;
  sh.nQb = block_mask ? (Tq + q_block - 1) / q_block : 0;
  sh.nKb = block_mask ? (Tk_max + k_block - 1) / k_block : 0;
  sh.timeout_ns = g_timeout_ns;

  // ---- fp32 storage: CUDA-core kernel (fp32 arithmetic throughout) -----------------------
  if (dtype == GA_F32) {
    dim3 grid((Tq + kSimtWarps - 1) / kSimtWarps, n_heads, batch);
    attend_simt_kernel<float><<<grid, 32 * kSimtWarps, 0, stream>>>(
        (const float*)q, (const float*)k, (const float*)v, (float*)out, lse, sh);
    return launch_status();
  }

  const __nv_bfloat16* qb = (const __nv_bfloat16*)q;
  __nv_bfloat16* ob = (__nv_bfloat16*)out;

  // ---- split-K decode ------------------------------------------------------------------
  if (decode_eligible(n_heads, n_kv, d, Tq, dtype, block_mask)) {
    DecodeShape ds{};
    ds.a = sh;
    ds.g = n_heads / n_kv;
    ds.rows = ds.g * Tq;
    ds.chunk_len = decode_chunk_len(batch, n_kv, Tk_max);
    ds.n_chunks = (Tk_max + ds.chunk_len - 1) / ds.chunk_len;
    if (ds.n_chunks == 1) ds.chunk_len = (Tk_max + 63) / 64 * 64;
    const size_t need = ga_workspace_size(batch, n_heads, n_kv, d, Tq, Tk_max, dtype);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
      return GA_ERR_WORKSPACE;
    float* ws_o = (float*)workspace;
    float* ws_ml = need ? ws_o + (size_t)batch * n_heads * Tq * ds.n_chunks * d : nullptr;
    CUtensorMap tk, tv;
    if (!make_map_bf16(&tk, k, d, Tk_max, (long long)batch * n_kv, 64) ||
        !make_map_bf16(&tv, v, d, Tk_max, (long long)batch * n_kv, 64))
      return GA_ERR_CUDA;
    return launch_decode(d, tk, tv, qb, ob, lse, ws_o, ws_ml, ds, stream);
  }

  // ---- tensor-core prefill ---------------------------------------------------------------
  if (tc_eligible(d, dtype, q, k, v, out, block_mask, q_block, k_block))
    return launch_prefill_tc(q, k, v, ob, lse, sh, block_mask != nullptr, WideEpi{0, nullptr, nullptr, 0.0f},
                             stream);

  // ---- everything else: CUDA-core kernel on bf16 storage --------------------------------
  dim3 grid((Tq + kSimtWarps - 1) / kSimtWarps, n_heads, batch);
  attend_simt_kernel<__nv_bfloat16><<<grid, 32 * kSimtWarps, 0, stream>>>(
      qb, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, ob, lse, sh);
  return launch_status();
}

int ga_attend_decode_static(const void* q, const void* k, const void* v, void* out, int batch,
                            int n_heads, int n_kv, int d, int Tq, int Tk_max, const int32_t* k_lens,
                            int causal, int window, const float* sink, float* lse,
                            ga_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  // ---- host-side checks, before any CUDA call -------------------------------------------
  if (!q || !k || !v || !out) return GA_ERR_INVALID_ARG;
  if (batch < 1 || n_heads < 1 || n_kv < 1 || n_kv > n_heads || n_heads % n_kv != 0)
    return GA_ERR_INVALID_ARG;
  if (d < 1 || d > 256 || Tq < 1 || Tk_max < Tq) return GA_ERR_INVALID_ARG;
  if ((causal != 0 && causal != 1) || window < 0 || (window > 0 && !causal)) return GA_ERR_INVALID_ARG;
  if (batch > 65535 || n_heads > 65535) return GA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (lse && !aligned16(lse)) || (sink && !aligned16(sink)) || (k_lens && !aligned16(k_lens)))
    return GA_ERR_INVALID_ARG;
  if (!decode_eligible(n_heads, n_kv, d, Tq, GA_BF16, nullptr)) return GA_ERR_UNSUPPORTED;
  const size_t need = ga_workspace_size(batch, n_heads, n_kv, d, Tq, Tk_max, GA_BF16);
  if (need > (size_t)GA_DECODE_STATIC_SCRATCH_BYTES) return GA_ERR_SCRATCH_LIMIT;

  // ---- once per device: the scratch array's device address -------------------------------
  void* scratch = nullptr;
  const int st0 = static_scratch_setup(&scratch);
  if (st0 != GA_OK) return st0;

  AttnShape sh{};
  sh.batch = batch; sh.n_heads = n_heads; sh.n_kv = n_kv; sh.d = d; sh.Tq = Tq; sh.Tk_max = Tk_max;
  sh.k_lens = k_lens; sh.causal = causal; sh.window = window; sh.sink = sink;
  sh.block_mask = nullptr; sh.q_block = 1; sh.k_block = 1; sh.nQb = 0; sh.nKb = 0;
  sh.timeout_ns = g_timeout_ns;
  DecodeShape ds{};
  ds.a = sh;
  ds.g = n_heads / n_kv;
  ds.rows = ds.g * Tq;
  ds.chunk_len = decode_chunk_len(batch, n_kv, Tk_max);
  ds.n_chunks = (Tk_max + ds.chunk_len - 1) / ds.chunk_len;
  if (ds.n_chunks == 1) ds.chunk_len = (Tk_max + 63) / 64 * 64;
  // partial rows first, then the (max, sum) pairs: the same layout as a caller's workspace
  float* ws_o = need ? static_cast<float*>(scratch) : nullptr;
  float* ws_ml = need ? ws_o + (size_t)batch * n_heads * Tq * ds.n_chunks * d : nullptr;
  const __nv_bfloat16* qb = (const __nv_bfloat16*)q;
  __nv_bfloat16* ob = (__nv_bfloat16*)out;
  CUtensorMap tk, tv;
  if (!make_map_bf16(&tk, k, d, Tk_max, (long long)batch * n_kv, 64) ||
      !make_map_bf16(&tv, v, d, Tk_max, (long long)batch * n_kv, 64))
    return GA_ERR_CUDA;
  return launch_decode(d, tk, tv, qb, ob, lse, ws_o, ws_ml, ds, stream);
}

int ga_attend_diff(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                   void* out, int batch, int n_heads, int n_kv, int d, int Tq, int Tk_max,
                   const int32_t* k_lens, int causal, int window, float lam, void* workspace,
                   size_t workspace_bytes, ga_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (!q1 || !k1 || !q2 || !k2 || !v || !out) return GA_ERR_INVALID_ARG;
  if (batch < 1 || n_heads < 1 || n_kv < 1 || n_kv > n_heads || n_heads % n_kv != 0)
    return GA_ERR_INVALID_ARG;
  if (Tq < 1 || Tk_max < Tq || !std::isfinite(lam)) return GA_ERR_INVALID_ARG;
  if ((causal != 0 && causal != 1) || window < 0 || (window > 0 && !causal)) return GA_ERR_INVALID_ARG;
  if (d != 128 && d != 256) return GA_ERR_UNSUPPORTED;
  if (batch > 65535 || n_heads > 65535) return GA_ERR_UNSUPPORTED;
  for (const void* p : {q1, k1, q2, k2, v, (const void*)out})
    if (!aligned16(p)) return GA_ERR_INVALID_ARG;
  if (k_lens && !aligned16(k_lens)) return GA_ERR_INVALID_ARG;
  const size_t need = (size_t)batch * n_heads * Tq * d * sizeof(float);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return GA_ERR_WORKSPACE;

  AttnShape sh{};
  sh.batch = batch; sh.n_heads = n_heads; sh.n_kv = n_kv; sh.d = d; sh.Tq = Tq; sh.Tk_max = Tk_max;
  sh.k_lens = k_lens; sh.causal = causal; sh.window = window; sh.sink = nullptr;
  sh.block_mask = nullptr; sh.q_block = 1; sh.k_block = 1; sh.nQb = 0; sh.nKb = 0;
  sh.timeout_ns = g_timeout_ns;
  float* a1v = static_cast<float*>(workspace);
  __nv_bfloat16* ob = (__nv_bfloat16*)out;
  // pass 1: A1 v in fp32; pass 2: out = A1 v - lam * A2 v, rounded once
  int st = launch_prefill_tc(q1, k1, v, ob, nullptr, sh, false, WideEpi{1, a1v, nullptr, 0.0f}, stream);
  if (st != GA_OK) return st;
  return launch_prefill_tc(q2, k2, v, ob, nullptr, sh, false, WideEpi{2, nullptr, a1v, lam}, stream);
}

int ga_dsa_indexer(const void* qi, const float* wi, const void* ki, const int32_t* lens, int batch,
                   int n_idx_heads, int di, int L_max, float* scores, ga_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (!qi || !wi || !ki || !scores || batch < 1 || L_max < 1) return GA_ERR_INVALID_ARG;
  if (!(di == 64 || di == 128) || n_idx_heads < 1 || n_idx_heads > di / 8 ||
      (n_idx_heads & (n_idx_heads - 1)) != 0)
    return GA_ERR_UNSUPPORTED;
  if (batch > 65535) return GA_ERR_UNSUPPORTED;
  if (!aligned16(qi) || !aligned16(ki) || (reinterpret_cast<uintptr_t>(wi) & 3) ||
      (reinterpret_cast<uintptr_t>(scores) & 3) || (lens && (reinterpret_cast<uintptr_t>(lens) & 3)))
    return GA_ERR_INVALID_ARG;
  const dim3 grid((L_max + kIdxWarps * kIdxKeysPerWarp - 1) / (kIdxWarps * kIdxKeysPerWarp), batch);
  const auto* q = (const __nv_bfloat16*)qi;
  const auto* kk = (const __nv_bfloat16*)ki;
#define GA_IDX(DI, HI) dsa_indexer_kernel<DI, HI><<<grid, 32 * kIdxWarps, 0, stream>>>(q, wi, kk, lens, L_max, scores)
  if (di == 128) {
    switch (n_idx_heads) {
      case 1: GA_IDX(128, 1); break;
      case 2: GA_IDX(128, 2); break;
      case 4: GA_IDX(128, 4); break;
      case 8: GA_IDX(128, 8); break;
      default: GA_IDX(128, 16); break;
    }
  } else {
    switch (n_idx_heads) {
      case 1: GA_IDX(64, 1); break;
      case 2: GA_IDX(64, 2); break;
      case 4: GA_IDX(64, 4); break;
      default: GA_IDX(64, 8); break;
    }
  }
#undef GA_IDX
  return launch_status();
}

int ga_topk_indices(const float* scores, const int32_t* lens, int batch, int L_max, int topk,
                    int32_t* idx, int32_t* n_sel, ga_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (!scores || !idx || !n_sel || batch < 1 || L_max < 1 || topk < 1) return GA_ERR_INVALID_ARG;
  if (batch > 0x7fffffff / 2) return GA_ERR_UNSUPPORTED;
  for (const void* p : {(const void*)scores, (const void*)idx, (const void*)n_sel, (const void*)lens})
    if (p && (reinterpret_cast<uintptr_t>(p) & 3)) return GA_ERR_INVALID_ARG;
  const DeviceKernels* dk = device_kernels();
  if (!dk) return GA_ERR_CUDA;
  if (L_max <= kTopkStageMax) {
    if (dk->topk != GA_OK) return dk->topk;
    // a programmatic dependent of the previous kernel (the indexer): its CTAs start launching
    // while the indexer's last ones run, and wait for it before reading the scores
    if (launch_pdl(topk_select_kernel<true>, dim3(batch), dim3(kTopkThreads), kTopkFixedSmem + (size_t)L_max * 4,
                   stream, scores, lens, L_max, topk, idx, n_sel) != cudaSuccess)
      return GA_ERR_CUDA;
  } else {
    if (dk->topk_unstaged != GA_OK) return dk->topk_unstaged;
    if (launch_pdl(topk_select_kernel<false>, dim3(batch), dim3(kTopkThreads), kTopkFixedSmem, stream, scores,
                   lens, L_max, topk, idx, n_sel) != cudaSuccess)
      return GA_ERR_CUDA;
  }
  return launch_status();
}

namespace {
// Key chunk of the gathered decode: about four CTAs per SM over the launch, at most
// kGatherMaxKeys keys, the selected keys split evenly into whole 64-key tiles.
int gather_chunk_len(int batch, int n_kv, int topk) {
  long long want = (long long)topk * batch * n_kv / (148LL * 4);
  want = want < 256 ? 256 : (want > kGatherMaxKeys ? kGatherMaxKeys : want);
  const long long n = (topk + want - 1) / want;
  return (int)(((topk + n - 1) / n + 63) / 64 * 64);
}
}  // namespace

size_t ga_attend_gather_workspace_size(int batch, int n_heads, int n_kv, int d, int topk) {
  if (batch < 1 || n_heads < 1 || n_kv < 1 || d < 1 || topk < 1 || n_heads % n_kv != 0) return SIZE_MAX;
  const int chunk = gather_chunk_len(batch, n_kv, topk);
  const size_t n_chunks = (topk + chunk - 1) / chunk;
  if (n_chunks <= 1) return 0;                  // one chunk writes the output itself
  return (size_t)batch * n_heads * n_chunks * (size_t)(d + 2) * sizeof(float);
}

int ga_attend_gather(const void* q, const void* k, const void* v, void* out, int batch, int n_heads,
                     int n_kv, int d, int Tk_max, const int32_t* idx, const int32_t* n_sel, int topk,
                     const float* sink, float* lse, void* workspace, size_t workspace_bytes,
                     ga_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (!q || !k || !v || !out || !idx || !n_sel || topk < 1 || Tk_max < 1) return GA_ERR_INVALID_ARG;
  if (batch < 1 || n_heads < 1 || n_kv < 1 || n_heads % n_kv != 0) return GA_ERR_INVALID_ARG;
  if (!(d == 64 || d == 128 || d == 256) || n_heads / n_kv > 16 || batch > 65535) return GA_ERR_UNSUPPORTED;
  if ((long long)batch * n_kv * Tk_max > 0x7fffffffLL) return GA_ERR_UNSUPPORTED;   // int32 row coordinates
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(n_sel) ||
      (reinterpret_cast<uintptr_t>(idx) & 3) || (lse && !aligned16(lse)) || (sink && !aligned16(sink)))
    return GA_ERR_INVALID_ARG;
  const size_t need = ga_attend_gather_workspace_size(batch, n_heads, n_kv, d, topk);
  if (need == SIZE_MAX) return GA_ERR_INVALID_ARG;
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return GA_ERR_WORKSPACE;
  // The query sees every selected token: a causal decode row over n_sel[b] keys, key j being
  // cache row idx[b, j] of the kv head.
  AttnShape sh{};
  sh.batch = batch; sh.n_heads = n_heads; sh.n_kv = n_kv; sh.d = d; sh.Tq = 1; sh.Tk_max = topk;
  sh.k_lens = n_sel; sh.causal = 1; sh.window = 0; sh.sink = sink;
  sh.block_mask = nullptr; sh.q_block = 1; sh.k_block = 1; sh.nQb = 0; sh.nKb = 0;
  sh.timeout_ns = g_timeout_ns;
  DecodeShape ds{};
  ds.a = sh;
  ds.g = n_heads / n_kv;
  ds.rows = ds.g;
  ds.chunk_len = gather_chunk_len(batch, n_kv, topk);
  ds.n_chunks = (topk + ds.chunk_len - 1) / ds.chunk_len;
  ds.gidx = idx; ds.gidx_stride = topk; ds.cache_T = Tk_max;
  ds.gk = (const __nv_bfloat16*)k; ds.gv = (const __nv_bfloat16*)v;
  if (ds.chunk_len > kGatherMaxKeys) return GA_ERR_UNSUPPORTED;    // not reached: chunks are <= 1024 keys
  float* ws_o = need ? static_cast<float*>(workspace) : nullptr;
  float* ws_ml = need ? ws_o + (size_t)batch * n_heads * ds.n_chunks * d : nullptr;
  CUtensorMap tk, tv;                             // not read by the gathered form
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  return launch_decode(d, tk, tv, (const __nv_bfloat16*)q, (__nv_bfloat16*)out, lse, ws_o, ws_ml, ds, stream,
                       /*gather=*/true);
}

namespace {
// CTAs of the MLA decode: two per SM.  The workspace is sized for kMlaMaxCta, so that it does
// not depend on the device it is used on.
constexpr int kMlaMaxCta = 2 * 192;

struct MlaWorkspace {
  __nv_bfloat16* q_abs;  // [batch, n_heads, 576]
  float* ws_o;           // [n_ids, n_heads, 512]
  float* ws_ml;          // [n_ids, n_heads, 2]
  int2* seg;             // [batch]
};

// Workspace layout (each part rounded up to 256 bytes); n_ids = kMlaMaxCta + batch - 1.
size_t mla_layout(int batch, int n_heads, void* base, MlaWorkspace* w) {
  using C = MlaCfg;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = (size_t)batch * n_heads, ids = (size_t)kMlaMaxCta + batch - 1;
  const size_t o_q = 0, o_o = o_q + up(rows * C::DK * 2), o_ml = o_o + up(ids * n_heads * C::R * 4),
               o_seg = o_ml + up(ids * n_heads * 2 * 4), total = o_seg + up((size_t)batch * 8);
  if (w) {
    unsigned char* p = static_cast<unsigned char*>(base);
    w->q_abs = reinterpret_cast<__nv_bfloat16*>(p + o_q);
    w->ws_o = reinterpret_cast<float*>(p + o_o);
    w->ws_ml = reinterpret_cast<float*>(p + o_ml);
    w->seg = reinterpret_cast<int2*>(p + o_seg);
  }
  return total;
}
}  // namespace

size_t ga_mla_decode_workspace_size(int batch, int n_heads, int L_max) {
  if (batch < 1 || n_heads < 1 || n_heads > 16 || L_max < 1) return SIZE_MAX;
  return mla_layout(batch, n_heads, nullptr, nullptr);
}

int ga_mla_decode(const void* q_nope, const void* q_rope, const void* latent, const void* w_uk,
                  const void* w_uv, const int32_t* lens, void* out, int batch, int n_heads, int L_max,
                  void* workspace, size_t workspace_bytes, ga_stream_t stream_) {
  using C = MlaCfg;
  cudaStream_t stream = (cudaStream_t)stream_;
  if (!q_nope || !q_rope || !latent || !w_uk || !w_uv || !out) return GA_ERR_INVALID_ARG;
  if (batch < 1 || n_heads < 1 || L_max < 1) return GA_ERR_INVALID_ARG;
  if (n_heads > 16 || batch > 65535 * C::EX_SEQ) return GA_ERR_UNSUPPORTED;
  for (const void* p : {q_nope, q_rope, latent, w_uk, w_uv, (const void*)out})
    if (!aligned16(p)) return GA_ERR_INVALID_ARG;
  if (lens && (reinterpret_cast<uintptr_t>(lens) & 3)) return GA_ERR_INVALID_ARG;
  const size_t need = ga_mla_decode_workspace_size(batch, n_heads, L_max);
  if (need == SIZE_MAX) return GA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return GA_ERR_WORKSPACE;
  MlaWorkspace w;
  mla_layout(batch, n_heads, workspace, &w);
  CUtensorMap tm;
  if (!make_map_bf16(&tm, latent, C::DK, L_max, batch, C::TILE)) return GA_ERR_CUDA;
  const DeviceKernels* dk = device_kernels();
  if (!dk) return GA_ERR_CUDA;
  if (dk->mla != GA_OK) return dk->mla;
  MlaShape s{};
  s.batch = batch; s.n_heads = n_heads; s.L_max = L_max; s.lens = lens; s.timeout_ns = g_timeout_ns;
  s.n_cta = 2 * dk->n_sm < kMlaMaxCta ? 2 * dk->n_sm : kMlaMaxCta;
  s.n_ids = s.n_cta + batch - 1;
  s.seg = w.seg;
  mla_absorb_kernel<<<dim3(C::R / C::AB_ROWS, n_heads, (batch + C::AB_SEQ - 1) / C::AB_SEQ), 128, 0, stream>>>(
      (const __nv_bfloat16*)q_nope, (const __nv_bfloat16*)q_rope, (const __nv_bfloat16*)w_uk, w.q_abs, n_heads,
      batch);
  // the decode streams its first latent tiles while the absorption finishes, the expansion
  // warms its weights while the decode finishes
  if (launch_pdl(mla_decode_kernel, dim3(s.n_cta), dim3(C::THREADS), C::SMEM_BYTES, stream, tm,
                 (const __nv_bfloat16*)w.q_abs, w.ws_o, w.ws_ml, s) != cudaSuccess)
    return GA_ERR_CUDA;
  if (launch_pdl(mla_expand_kernel, dim3(C::DV / C::EX_DIMS, n_heads, (batch + C::EX_SEQ - 1) / C::EX_SEQ), dim3(256),
                 C::EX_SMEM, stream, (const float*)w.ws_o, (const float*)w.ws_ml, (const __nv_bfloat16*)w_uv,
                 (__nv_bfloat16*)out, s) != cudaSuccess)
    return GA_ERR_CUDA;
  return launch_status();
}

int ga_ring_append(void* k_ring, void* v_ring, const void* k_new, const void* v_new, int32_t* n_seen,
                   int batch, int n_kv, int d, int W, ga_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (!k_ring || !v_ring || !k_new || !v_new || !n_seen) return GA_ERR_INVALID_ARG;
  if (batch < 1 || n_kv < 1 || W < 1 || d < 8 || d > 256 || d % 8 != 0) return GA_ERR_INVALID_ARG;
  if (batch > 0x7fffffff / 2) return GA_ERR_UNSUPPORTED;
  if (!aligned16(k_ring) || !aligned16(v_ring) || !aligned16(k_new) || !aligned16(v_new) ||
      (reinterpret_cast<uintptr_t>(n_seen) & 3) != 0)
    return GA_ERR_INVALID_ARG;
  ring_append_kernel<<<batch, kRingThreads, 0, stream>>>(
      (__nv_bfloat16*)k_ring, (__nv_bfloat16*)v_ring, (const __nv_bfloat16*)k_new,
      (const __nv_bfloat16*)v_new, n_seen, n_kv, d, W);
  return launch_status();
}

int ga_attend_ring(const void* q, const void* k_ring, const void* v_ring, void* out, int batch,
                   int n_heads, int n_kv, int d, int W, const int32_t* n_seen, const float* sink,
                   float* lse, void* workspace, size_t workspace_bytes, ga_stream_t stream) {
  if (!n_seen || W < 1 || n_heads < 1 || n_kv < 1 || n_heads % n_kv != 0) return GA_ERR_INVALID_ARG;
  if (!(d == 64 || d == 128 || d == 256) || n_heads / n_kv > 16) return GA_ERR_UNSUPPORTED;
  // The query is the newest token, at absolute position n_seen - 1 of its sequence; with a
  // window of W positions the keys it may use are exactly the min(n_seen, W) filled slots.
  // Over the ring that is a causal decode row whose key count is n_seen clamped to W (the
  // kernels clamp every length to [0, Tk_max] = [0, W]).
  return ga_attend(q, k_ring, v_ring, out, batch, n_heads, n_kv, d, 1, W, n_seen, 1, 0, sink, nullptr,
                   1, 1, lse, GA_BF16, workspace, workspace_bytes, stream);
}

int ga_block_stats(const void* k, const int32_t* k_lens, int batch, int n_kv, int d, int Tk_max,
                   int k_block, float* centroid, float* radius, ga_dtype dtype, ga_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (!k || !centroid || !radius) return GA_ERR_INVALID_ARG;
  if (dtype != GA_F32 && dtype != GA_BF16) return GA_ERR_INVALID_ARG;
  if (batch < 1 || n_kv < 1 || d < 1 || d > 256 || Tk_max < 1 || k_block < 1 || k_block > 1024)
    return GA_ERR_INVALID_ARG;
  if (batch > 65535 || n_kv > 65535) return GA_ERR_UNSUPPORTED;
  if (!aligned16(k) || !aligned16(centroid) || !aligned16(radius) || (k_lens && !aligned16(k_lens)))
    return GA_ERR_INVALID_ARG;
  const int nKb = (Tk_max + k_block - 1) / k_block;
  if (dtype == GA_BF16 && d % 8 == 0 && 32 % (d / 8) == 0) {
    const long long n_blk = (long long)batch * n_kv * nKb;
    const long long n_cta = (n_blk + kStatsVecWarps - 1) / kStatsVecWarps;
    if (n_cta > 0x7fffffffLL) return GA_ERR_UNSUPPORTED;
    const dim3 vgrid((unsigned)n_cta);
    const __nv_bfloat16* kp = (const __nv_bfloat16*)k;
    if (k_block <= 64 && (d == 32 || d == 64 || d == 128)) {   // block held in registers: one read
      const auto kern = d == 32 ? block_stats_reg_kernel<4>
                      : d == 64 ? block_stats_reg_kernel<8>
                                : block_stats_reg_kernel<16>;
      kern<<<vgrid, 32 * kStatsVecWarps, 0, stream>>>(kp, k_lens, batch, n_kv, Tk_max, k_block, nKb, centroid,
                                                      radius);
      return launch_status();
    }
    switch (d / 8) {
      case 1: block_stats_vec_kernel<1><<<vgrid, 32 * kStatsVecWarps, 0, stream>>>(kp, k_lens, batch, n_kv, Tk_max, k_block, nKb, centroid, radius); break;
      case 2: block_stats_vec_kernel<2><<<vgrid, 32 * kStatsVecWarps, 0, stream>>>(kp, k_lens, batch, n_kv, Tk_max, k_block, nKb, centroid, radius); break;
      case 4: block_stats_vec_kernel<4><<<vgrid, 32 * kStatsVecWarps, 0, stream>>>(kp, k_lens, batch, n_kv, Tk_max, k_block, nKb, centroid, radius); break;
      case 8: block_stats_vec_kernel<8><<<vgrid, 32 * kStatsVecWarps, 0, stream>>>(kp, k_lens, batch, n_kv, Tk_max, k_block, nKb, centroid, radius); break;
      case 16: block_stats_vec_kernel<16><<<vgrid, 32 * kStatsVecWarps, 0, stream>>>(kp, k_lens, batch, n_kv, Tk_max, k_block, nKb, centroid, radius); break;
      default: block_stats_vec_kernel<32><<<vgrid, 32 * kStatsVecWarps, 0, stream>>>(kp, k_lens, batch, n_kv, Tk_max, k_block, nKb, centroid, radius); break;
    }
    return launch_status();
  }
  dim3 grid(nKb, n_kv, batch);
  if (dtype == GA_BF16)
    block_stats_kernel<__nv_bfloat16><<<grid, kStatsThreads, 0, stream>>>(
        (const __nv_bfloat16*)k, k_lens, n_kv, d, Tk_max, k_block, nKb, centroid, radius);
  else
    block_stats_kernel<float><<<grid, kStatsThreads, 0, stream>>>((const float*)k, k_lens, n_kv, d,
                                                                  Tk_max, k_block, nKb, centroid, radius);
  return launch_status();
}

namespace {
// Workspace of the selection: pooled query rows and centroids split into high and low parts
// (rows of d rounded up to 32), the rows' norms, the row maxima, the rescue flags and the
// mean-branch scores, each part 256-byte aligned.
struct SelectWs {
  size_t q_hi, q_lo, c_hi, c_lo, qnorm, rowmax, rescue, scores, total;
};
SelectWs select_ws(int batch, int n_hp, int n_kv, int d, int nQb, int nKb) {
  SelectWs w;
  const int dp = (d + 31) / 32 * 32;
  const size_t qb = sel_up256((size_t)batch * n_hp * nQb * dp * 4), cb = sel_up256((size_t)batch * n_kv * nKb * dp * 4);
  w.q_hi = 0;
  w.q_lo = w.q_hi + qb;
  w.c_hi = w.q_lo + qb;
  w.c_lo = w.c_hi + cb;
  w.qnorm = w.c_lo + cb;
  w.rowmax = w.qnorm + sel_up256((size_t)batch * n_hp * nQb * 4);
  w.rescue = w.rowmax + sel_up256((size_t)batch * n_hp * nQb * 4);
  w.scores = w.rescue + sel_up256((size_t)batch * n_kv * nKb);
  w.total = w.scores + sel_up256((size_t)batch * n_hp * nQb * sel_score_stride(nKb) * 4);
  return w;
}
}  // namespace

size_t ga_select_workspace_size(int batch, int n_heads, int n_kv, int d, int Tq, int Tk, int q_block,
                                int k_block, int group_shared) {
  if (batch < 1 || n_heads < 1 || n_kv < 1 || n_kv > n_heads || n_heads % n_kv != 0 || d < 1 || d > 256 ||
      Tq < 1 || Tk < Tq || q_block < 1 || k_block < 1 || (group_shared != 0 && group_shared != 1))
    return SIZE_MAX;
  const int nQb = (Tq + q_block - 1) / q_block;
  const int nKb = (int)(((long long)Tk + k_block - 1) / k_block);
  return select_ws(batch, group_shared ? n_kv : n_heads, n_kv, d, nQb, nKb).total;
}

int ga_select_blocks(const void* q, const float* centroid, const float* radius, int batch,
                     int n_heads, int n_kv, int d, int Tq, int Tk, int nKb_out, int q_block,
                     int k_block, int causal, int window, float tau_mean, float lambda_radius,
                     uint8_t* block_mask, int32_t* n_selected, ga_dtype dtype, void* workspace,
                     size_t workspace_bytes, ga_stream_t stream_) {
  return ga_select_blocks_ex(q, centroid, radius, batch, n_heads, n_kv, d, Tq, Tk, nKb_out, q_block,
                             k_block, causal, window, tau_mean, lambda_radius, GA_RADIUS_ZSCORE,
                             -INFINITY, 0, block_mask, n_selected, dtype, workspace, workspace_bytes, stream_);
}

int ga_select_blocks_ex(const void* q, const float* centroid, const float* radius, int batch,
                        int n_heads, int n_kv, int d, int Tq, int Tk, int nKb_out, int q_block,
                        int k_block, int causal, int window, float tau_mean, float lambda_radius,
                        int radius_rule, float tau_bound, int group_shared, uint8_t* block_mask,
                        int32_t* n_selected, ga_dtype dtype, void* workspace, size_t workspace_bytes,
                        ga_stream_t stream_) {
  cudaStream_t stream = (cudaStream_t)stream_;
  if (!q || !centroid || !radius || !block_mask) return GA_ERR_INVALID_ARG;
  if (dtype != GA_F32 && dtype != GA_BF16) return GA_ERR_INVALID_ARG;
  if (batch < 1 || n_heads < 1 || n_kv < 1 || n_kv > n_heads || n_heads % n_kv != 0)
    return GA_ERR_INVALID_ARG;
  if (d < 1 || d > 256 || Tq < 1 || Tk < Tq || q_block < 1 || q_block > 4096 || k_block < 1)
    return GA_ERR_INVALID_ARG;
  if ((causal != 0 && causal != 1) || window < 0 || (window > 0 && !causal)) return GA_ERR_INVALID_ARG;
  if (std::isnan(tau_mean) || std::isnan(lambda_radius) || std::isnan(tau_bound)) return GA_ERR_INVALID_ARG;
  if (radius_rule != GA_RADIUS_ZSCORE && radius_rule != GA_RADIUS_MAD) return GA_ERR_INVALID_ARG;
  if (group_shared != 0 && group_shared != 1) return GA_ERR_INVALID_ARG;
  const long long nKb = ((long long)Tk + k_block - 1) / k_block;
  if (nKb_out < nKb) return GA_ERR_INVALID_ARG;
  if (nKb > 32768 || batch > 65535 || n_heads > 65535) return GA_ERR_UNSUPPORTED;
  if (radius_rule == GA_RADIUS_MAD && nKb > 16384) return GA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(centroid) || !aligned16(radius)) return GA_ERR_INVALID_ARG;
  if (n_selected && (reinterpret_cast<uintptr_t>(n_selected) & 3)) return GA_ERR_INVALID_ARG;
  const int n_hp = group_shared ? n_kv : n_heads;
  const int nQb = (Tq + q_block - 1) / q_block;
  const SelectWs ws = select_ws(batch, n_hp, n_kv, d, nQb, (int)nKb);
  if (!workspace || workspace_bytes < ws.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return GA_ERR_WORKSPACE;
  if ((long long)batch * n_hp > 65535 || nQb > 0x7fffffff / 2) return GA_ERR_UNSUPPORTED;

  SelectShape s{};
  s.batch = batch; s.n_heads = n_heads; s.n_kv = n_kv; s.d = d; s.Tq = Tq; s.Tk = Tk;
  s.nKb_out = nKb_out; s.q_block = q_block; s.k_block = k_block; s.causal = causal;
  s.window = window; s.nQb = nQb; s.nKb = (int)nKb;
  s.tau_mean = tau_mean; s.lambda_radius = lambda_radius;
  s.radius_rule = radius_rule; s.tau_bound = tau_bound; s.group_shared = group_shared;
  s.n_hp = n_hp;
  s.sort_len = 0;
  if (radius_rule == GA_RADIUS_MAD)
    for (s.sort_len = 1; s.sort_len < nKb; s.sort_len <<= 1) {}
  unsigned char* w = static_cast<unsigned char*>(workspace);
  s.dp = (d + 31) / 32 * 32;
  s.q_hi = reinterpret_cast<float*>(w + ws.q_hi);
  s.q_lo = reinterpret_cast<float*>(w + ws.q_lo);
  s.c_hi = reinterpret_cast<float*>(w + ws.c_hi);
  s.c_lo = reinterpret_cast<float*>(w + ws.c_lo);
  s.timeout_ns = g_timeout_ns;
  s.qnorm = reinterpret_cast<float*>(w + ws.qnorm);
  s.rowmax = reinterpret_cast<int*>(w + ws.rowmax);
  s.rescue = w + ws.rescue;
  s.scores = reinterpret_cast<float*>(w + ws.scores);
  const DeviceKernels* dk = device_kernels();
  if (!dk) return GA_ERR_CUDA;
  if (dk->select != GA_OK) return dk->select;

  CUtensorMap tm_qh, tm_ql, tm_ch, tm_cl;
  const long long q_rows = (long long)batch * n_hp * nQb, c_rows = (long long)batch * n_kv * nKb;
  if (q_rows > 0x7fffffffLL || c_rows > 0x7fffffffLL) return GA_ERR_UNSUPPORTED;
  if (!make_map_f32(&tm_qh, s.q_hi, s.dp, q_rows, 1, kScA) || !make_map_f32(&tm_ql, s.q_lo, s.dp, q_rows, 1, kScA) ||
      !make_map_f32(&tm_ch, s.c_hi, s.dp, c_rows, 1, kScB) || !make_map_f32(&tm_cl, s.c_lo, s.dp, c_rows, 1, kScB))
    return GA_ERR_CUDA;
  // columns: nQb pooled query blocks, the z-score radius branch, then the centroid splits
  const int n_ct = (int)((nKb + kScB - 1) / kScB);
  const dim3 pool_grid(nQb + 1 + n_ct, n_hp, batch);
  if (dtype == GA_BF16)
    select_pool_kernel<__nv_bfloat16><<<pool_grid, kPoolThreads, 0, stream>>>((const __nv_bfloat16*)q, radius,
                                                                               centroid, s);
  else
    select_pool_kernel<float><<<pool_grid, kPoolThreads, 0, stream>>>((const float*)q, radius, centroid, s);
  // the later launches are programmatic dependents of the one before: each starts launching (and
  // the score kernel its set-up) while its predecessor finishes, and waits on it before reading
  if (radius_rule == GA_RADIUS_MAD &&
      launch_pdl(select_rescue_kernel, dim3(n_kv, batch), dim3(kRescueThreads), (size_t)s.sort_len * 8, stream, radius,
                 s) != cudaSuccess)
    return GA_ERR_CUDA;
  // persistent: one CTA per SM (or per tile when there are fewer tiles)
  const long long n_tiles = sel_score_tiles(batch, n_hp, nQb, (int)nKb);
  if (launch_pdl(select_score_kernel, dim3((unsigned)(n_tiles < dk->n_sm ? n_tiles : dk->n_sm)), dim3(kScThreads),
                 kScSmem, stream, tm_qh, tm_ql, tm_ch, tm_cl, s) != cudaSuccess)
    return GA_ERR_CUDA;
  const long long n_rows = (long long)batch * n_hp * nQb;
  if (launch_pdl(select_decide_kernel, dim3((unsigned)((n_rows + kDecWarps - 1) / kDecWarps)), dim3(32 * kDecWarps), 0,
                 stream, radius, block_mask, n_selected, s) != cudaSuccess)
    return GA_ERR_CUDA;
  return launch_status();
}

}  // extern "C"
