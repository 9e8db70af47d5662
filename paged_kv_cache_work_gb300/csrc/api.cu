// The C ABI declared in include/pa.h: host-side validation, the kernel variant for a
// configuration, the TMA descriptors of the two caches, and the stream-ordered launches.
// Nothing here allocates, synchronises (except pa_read_flags) or aborts.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "pa_internal.cuh"

using namespace pa;

namespace {

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape and type checks that need no device.  Unsupported-but-well-formed configurations
// (head dim, page size, dtype combination, head grouping) map to PA_ERR_UNSUPPORTED, as the
// block-size and dtype rejection cases of "Optimize paged-attention metadata decode"
// (FlyDSL PR #910, validation coverage) do; malformed values to PA_ERR_INVALID_ARG.
pa_status validate(const pa_config* c) {
  if (!c) return PA_ERR_INVALID_ARG;
  if (c->batch < 1 || c->max_q_len < 1 || c->num_q_heads < 1 || c->num_kv_heads < 1 ||
      c->max_blocks_per_seq < 1 || c->num_blocks < 1 || c->head_dim < 1 || c->block_size < 1)
    return PA_ERR_INVALID_ARG;
  if (c->q_dtype < PA_BF16 || c->q_dtype > PA_FP8_E4M3 || c->kv_dtype < PA_BF16 ||
      c->kv_dtype > PA_FP8_E4M3)
    return PA_ERR_INVALID_ARG;
  if (c->kv_scale_mode < PA_SCALE_NONE || c->kv_scale_mode > PA_SCALE_PER_TOKEN)
    return PA_ERR_INVALID_ARG;
  if (c->causal != 0 && c->causal != 1) return PA_ERR_INVALID_ARG;
  if (!std::isfinite(c->sm_scale)) return PA_ERR_INVALID_ARG;
  if (c->num_ctas < 0 || c->grid_mult < 0) return PA_ERR_INVALID_ARG;
  if (c->split_merge < PA_MERGE_AUTO || c->split_merge > PA_MERGE_IN_REDUCE)
    return PA_ERR_INVALID_ARG;
  if (c->num_q_heads % c->num_kv_heads != 0) return PA_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(c->block_size) || c->block_size < 16 || c->block_size > 1024)
    return PA_ERR_UNSUPPORTED;
  if (c->q_dtype != PA_BF16 && c->q_dtype != PA_FP16) return PA_ERR_UNSUPPORTED;
  if (c->kv_dtype != c->q_dtype && c->kv_dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
  if (c->kv_dtype != PA_FP8_E4M3 && c->kv_scale_mode != PA_SCALE_NONE) return PA_ERR_UNSUPPORTED;
  const long long rows = (long long)(c->num_q_heads / c->num_kv_heads) * c->max_q_len;
  if (rows > (1 << 20)) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// Persistent grid: num_ctas if given, else (SMs x grid_mult) x the decode CTAs that fit
// on one SM: one resident wave at multiplier 1; with a larger one the later CTAs start as
// earlier ones finish.
pa_status resolve_ctas(const pa_config& c, Variant* v) {
  if (c.num_ctas > 0) {
    v->ctas = c.num_ctas > 65535 ? 65535 : c.num_ctas;
    return PA_OK;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PA_ERR_CUDA;
  v->sms = sms;
  const int mult = c.grid_mult > 0 ? c.grid_mult : 1;
  long long n = (long long)sms * mult * v->ctas_per_sm;
  v->ctas = (int)(n > 65535 ? 65535 : n);
  return PA_OK;
}

pa_status prepare(const pa_config* cfg, Variant* v, WsLayout* L) {
  pa_status st = validate(cfg);
  if (st != PA_OK) return st;
  *v = make_variant(*cfg);
  st = resolve_ctas(*cfg, v);
  if (st != PA_OK) return st;
  // The planner's concatenated token space is indexed with int32.
  const long long per_unit =
      (long long)cfg->max_blocks_per_seq * cfg->block_size + v->tt + v->item_cost;
  if ((long long)v->units * per_unit >= (1ll << 30)) return PA_ERR_UNSUPPORTED;
  *L = ws_layout(*cfg, *v);
  return PA_OK;
}

pa_status check_ws(const void* ws, size_t ws_bytes, const WsLayout& L) {
  if (!ws || !aligned(ws, 256)) return PA_ERR_INVALID_ARG;
  if (ws_bytes < L.total) return PA_ERR_WORKSPACE;
  return PA_OK;
}

ProblemArgs problem_args(const pa_config& c, const int32_t* bt, const int32_t* ctx,
                         const int32_t* ql) {
  ProblemArgs a;
  a.block_tables = bt;
  a.context_lens = ctx;
  a.q_lens = ql;
  a.batch = c.batch;
  a.max_q_len = c.max_q_len;
  a.num_q_heads = c.num_q_heads;
  a.num_kv_heads = c.num_kv_heads;
  a.head_dim = c.head_dim;
  a.block_size = c.block_size;
  a.max_blocks = c.max_blocks_per_seq;
  a.num_blocks = c.num_blocks;
  a.causal = c.causal;
  return a;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the library does not
// link libcuda directly.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Descriptor of a cache [num_blocks, block_size, Hkv, D] seen as a 4-D tensor (D innermost)
// with a box of one head's rows of one page.  CUDA-core kernel: {D, 1, rows, 1}, no swizzle.
// Tensor-core kernel: {128 bytes of D, 1, rows, 1} with the 128-byte swizzle, one box per
// 128-byte column slab.
bool kv_tensor_map(CUtensorMap* m, const void* base, const pa_config& c, int box_rows, bool slabs) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const int bpe = c.kv_dtype == PA_FP8_E4M3 ? 1 : 2;
  CUtensorMapDataType dt = c.kv_dtype == PA_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                           : c.kv_dtype == PA_FP16   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[4] = {(cuuint64_t)c.head_dim, (cuuint64_t)c.num_kv_heads,
                        (cuuint64_t)c.block_size, (cuuint64_t)c.num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)c.head_dim * bpe,
                           (cuuint64_t)c.num_kv_heads * c.head_dim * bpe,
                           (cuuint64_t)c.block_size * c.num_kv_heads * c.head_dim * bpe};
  const cuuint32_t inner = slabs ? (cuuint32_t)(128 / bpe) : (cuuint32_t)c.head_dim;
  cuuint32_t box[4] = {inner, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  std::memset(m, 0, sizeof(*m));
  CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   slabs ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

pa_status pa_workspace_size(const pa_config* cfg, size_t* bytes) {
  if (!cfg || !bytes) return PA_ERR_INVALID_ARG;
  Variant v;
  WsLayout L;
  pa_status st = prepare(cfg, &v, &L);
  if (st != PA_OK) return st;
  *bytes = L.total;
  return PA_OK;
}

pa_status pa_plan(const pa_config* cfg, const int32_t* block_tables, const int32_t* context_lens,
                  const int32_t* q_lens, void* ws, size_t ws_bytes, pa_stream stream) {
  Variant v;
  WsLayout L;
  pa_status st = prepare(cfg, &v, &L);
  if (st != PA_OK) return st;
  if (!block_tables || !context_lens || !q_lens) return PA_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, L)) != PA_OK) return st;
  const ProblemArgs a = problem_args(*cfg, block_tables, context_lens, q_lens);
  if (launch_plan(a, v, L, static_cast<char*>(ws), reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

pa_status pa_decode(const pa_config* cfg, const void* q, const void* k_cache, const void* v_cache,
                    const float* k_scale, const float* v_scale, const int32_t* block_tables,
                    const int32_t* context_lens, const int32_t* q_lens, void* out, float* lse,
                    void* ws, size_t ws_bytes, pa_stream stream) {
  Variant v;
  WsLayout L;
  pa_status st = prepare(cfg, &v, &L);
  if (st != PA_OK) return st;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !q_lens || !out)
    return PA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return PA_ERR_INVALID_ARG;
  if (lse && !aligned(lse, 4)) return PA_ERR_INVALID_ARG;
  if (cfg->kv_scale_mode != PA_SCALE_NONE) {
    if (!k_scale || !v_scale || !aligned(k_scale, 4) || !aligned(v_scale, 4))
      return PA_ERR_INVALID_ARG;
  }
  if ((st = check_ws(ws, ws_bytes, L)) != PA_OK) return st;

  const int box_rows = cfg->block_size < v.tt ? cfg->block_size : v.tt;
  CUtensorMap kmap, vmap;
  if (!kv_tensor_map(&kmap, k_cache, *cfg, box_rows, v.path >= 1) ||
      !kv_tensor_map(&vmap, v_cache, *cfg, box_rows, v.path >= 1))
    return PA_ERR_CUDA;

  DecodeArgs a;
  a.p = problem_args(*cfg, block_tables, context_lens, q_lens);
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.scale_mode = cfg->kv_scale_mode;
  a.qk_scale = cfg->sm_scale * kLog2e;
  a.out = out;
  a.lse = lse;
  a.ws = static_cast<char*>(ws);
  a.L = L;
  a.v = v;
  a.q_kind = cfg->q_dtype == PA_FP16 ? Q_FP16 : Q_BF16;
  a.kv_kind = cfg->kv_dtype == PA_FP8_E4M3 ? KV_FP8 : cfg->kv_dtype == PA_FP16 ? KV_FP16 : KV_BF16;
  cudaError_t e = launch_decode(a, kmap, vmap, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_reduce(const pa_config* cfg, void* out, float* lse, void* ws, size_t ws_bytes,
                    pa_stream stream) {
  Variant v;
  WsLayout L;
  pa_status st = prepare(cfg, &v, &L);
  if (st != PA_OK) return st;
  if (!out || !aligned(out, 16)) return PA_ERR_INVALID_ARG;
  if (lse && !aligned(lse, 4)) return PA_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, L)) != PA_OK) return st;
  if (cfg->split_merge == PA_MERGE_IN_DECODE) return PA_OK;  // pa_decode finished the step
  DecodeArgs a{};
  a.p = problem_args(*cfg, nullptr, nullptr, nullptr);
  a.out = out;
  a.lse = lse;
  a.ws = static_cast<char*>(ws);
  a.L = L;
  a.v = v;
  a.q_kind = cfg->q_dtype == PA_FP16 ? Q_FP16 : Q_BF16;
  return launch_reduce(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                : PA_ERR_CUDA;
}

pa_status pa_read_flags(const void* ws, size_t ws_bytes, int32_t* flags, pa_stream stream) {
  if (!ws || !flags || !aligned(ws, 256) || ws_bytes < 64 * sizeof(int32_t))
    return PA_ERR_INVALID_ARG;
  int32_t host = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&host, static_cast<const char*>(ws) + HDR_FLAGS * sizeof(int32_t),
                      sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  *flags = host;
  return host ? PA_ERR_DEVICE : PA_OK;
}

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_WORKSPACE: return "workspace too small";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_DEVICE: return "device-side input problem (see flags)";
    default: return "unknown status";
  }
}

}  // extern "C"
