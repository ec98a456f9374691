// libpagedkv: C ABI (include/pagedkv.h) over the sm_103a kernels.
//
// Host side only: argument validation, launch planning, TMA tensor-map
// encoding and kernel launches.  Nothing here allocates device memory.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "pkv_attention_simt.cuh"
#include "pkv_attention_tc.cuh"
#include "pkv_prefill.cuh"
#include "pkv_prefill_tc05.cuh"
#include "pkv_prefill_tc05x2.cuh"
#include "pkv_reduce.cuh"
#include "pkv_copy.cuh"
#include "pkv_device.cuh"

namespace {

thread_local std::string g_last_msg;

pkv_status fail(pkv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_msg = buf;
  return st;
}

#define PKV_CUDA(call)                                                                 \
  do {                                                                                 \
    cudaError_t e_ = (call);                                                           \
    if (e_ != cudaSuccess) return fail(PKV_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

#define PKV_CHECK(cond, st, ...)                  \
  do {                                            \
    if (!(cond)) return fail((st), __VA_ARGS__);  \
  } while (0)

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline size_t elem_bytes(pkv_dtype d) { return d == PKV_BF16 ? 2 : 4; }
inline bool dtype_ok(pkv_dtype d) { return d == PKV_F32 || d == PKV_BF16; }
inline int log2_exact(int64_t x) {
  if (x <= 0 || (x & (x - 1))) return -1;
  int l = 0;
  while ((int64_t(1) << l) < x) ++l;
  return l;
}

// ---- per-device facts --------------------------------------------------------
constexpr int kMaxDevices = 64;
struct DeviceFacts {
  std::once_flag once;
  int sm_count = 0;
  cudaError_t err = cudaSuccess;
};
DeviceFacts g_dev[kMaxDevices];

pkv_status device_facts(int* dev_out, int* sm_count) {
  int dev = 0;
  PKV_CUDA(cudaGetDevice(&dev));
  PKV_CHECK(dev >= 0 && dev < kMaxDevices, PKV_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
  DeviceFacts& f = g_dev[dev];
  std::call_once(f.once, [&] {
    f.err = cudaDeviceGetAttribute(&f.sm_count, cudaDevAttrMultiProcessorCount, dev);
  });
  if (f.err != cudaSuccess) return fail(PKV_ERR_CUDA, "SM count: %s", cudaGetErrorString(f.err));
  *dev_out = dev;
  *sm_count = f.sm_count;
  return PKV_OK;
}

// Opt a kernel into large dynamic shared memory once per device.
template <typename Kernel>
pkv_status set_smem_once(Kernel k, int bytes, std::once_flag (&flags)[kMaxDevices],
                         cudaError_t (&errs)[kMaxDevices], int dev) {
  std::call_once(flags[dev], [&] {
    errs[dev] = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  });
  if (errs[dev] != cudaSuccess)
    return fail(PKV_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(errs[dev]));
  return PKV_OK;
}

// ---- driver entry point for tensor maps -------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

pkv_status get_encode(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  PKV_CHECK(g_encode != nullptr, PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  *fn = g_encode;
  return PKV_OK;
}

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel in the stream finishes; it waits for that
// kernel's results (griddepcontrol.wait) before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
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

// ---- attention planning -------------------------------------------------------
enum { KIND_TC = 1, KIND_SIMT = 2 };

struct AttnPlan {
  int kind = 0;
  int hpc = 0, groups = 0, n_per_group = 0;  // tensor-core kernel
  int ps = 0;                                // CUDA-core kernel: tokens per partition
  int share_m = 1;                           // tensor-core kernel: sequences per shared-prefix group
  int pmax = 1;                              // partials per row (CUDA-core / multi-query layout)
  int64_t slots = 0;                         // partial slots of the workspace
  int64_t slot_stride = 0;                   // tensor-core kernel: slots per member region
  bool reduce = false;                       // a split-K reduce launch follows
  int seq_batch = 0;
  size_t ws_bytes = 0;
};

bool tc_shape_ok(int G, int D, int K, int64_t num_blocks, pkv_dtype dt) {
  return dt == PKV_BF16 && (D == 64 || D == 128) && G >= 1 && G <= 8 && (K % 16 == 0 || K == 8) &&
         num_blocks * K < (int64_t(1) << 31) - 64;
}

bool simt_shape_ok(int G, int D) {
  return (D == 32 || D == 64 || D == 128 || D == 256) && G >= 1 && G <= 16;
}

int tc_hpc(int H_kv) {
  for (int h : {8, 4, 2, 1})
    if (H_kv % h == 0) return h;
  return 1;
}

// Workspace layout of a decode plan: meta (one int4 per row of a launch
// batch), the partial (m, l) pairs and outputs per slot, then (shared-prefix
// groups) the groups' shared lengths.
struct WsLayout {
  size_t ml, o, glen, total;
};
WsLayout ws_layout(const AttnPlan& p, int H_q, int H_kv, int D) {
  const size_t sb = (size_t)std::max(p.seq_batch, 1);
  WsLayout l;
  l.ml = align256(sb * sizeof(int4));
  l.o = l.ml + align256((size_t)p.slots * H_q * sizeof(float2));
  l.glen = l.o + align256((size_t)p.slots * H_q * (size_t)D * sizeof(float));
  l.total = l.glen + (p.share_m > 1 ? align256(ceil_div((int64_t)sb, p.share_m) * 4) : 0);
  (void)H_kv;
  return l;
}

pkv_status plan_attention(int S, int H_q, int H_kv, int D, int K, int max_len, int64_t num_blocks,
                          pkv_dtype dt, const pkv_attention_config* cfg, bool tma_aligned,
                          AttnPlan* plan) {
  PKV_CHECK(S >= 0 && H_q > 0 && H_kv > 0 && D > 0 && K > 0 && K <= 1024 && max_len >= 0,
            PKV_ERR_INVALID_ARGUMENT, "bad attention sizes");
  PKV_CHECK(H_q % H_kv == 0, PKV_ERR_INVALID_ARGUMENT, "num_q_heads %% num_kv_heads != 0");
  PKV_CHECK(dtype_ok(dt), PKV_ERR_INVALID_ARGUMENT, "bad dtype");
  pkv_attention_config c = {};
  if (cfg) c = *cfg;
  for (int r : c.reserved) PKV_CHECK(r == 0, PKV_ERR_INVALID_ARGUMENT, "reserved config fields must be 0");
  PKV_CHECK(c.kernel >= 0 && c.kernel <= 2 && c.num_splits >= 0 &&
                (c.share_prefix == 0 || c.share_prefix == 1),
            PKV_ERR_INVALID_ARGUMENT, "bad attention config");
  const int G = H_q / H_kv;
  const bool tc_ok = tc_shape_ok(G, D, K, num_blocks, dt) && tma_aligned;
  AttnPlan p;
  if (c.kernel == 1 || (c.kernel == 0 && tc_ok)) {
    PKV_CHECK(tc_ok, PKV_ERR_UNSUPPORTED,
              "tensor-core kernel needs bf16, head_dim 64/128, G <= 8, block_size 8 or a multiple of 16 "
              "and a 16-byte aligned pool");
    int dev, sms;
    pkv_status st = device_facts(&dev, &sms);
    if (st != PKV_OK) return st;
    p.kind = KIND_TC;
    p.hpc = tc_hpc(H_kv);
    p.groups = H_kv / p.hpc;
    const int total = sms;   // one CTA per SM (shared memory bound)
    p.n_per_group = c.num_splits ? c.num_splits : (total / p.groups > 0 ? total / p.groups : 1);
    const int max_chunks = (int)ceil_div(max_len, pkv::kTcChunk);
    p.pmax = std::max(1, std::min(p.n_per_group, max_chunks));
    p.seq_batch = std::min(S, pkv::kTcMaxSeqs);
    if (c.share_prefix && G <= 8) {
      // groups of 16 / G sequences fill the kernel's two 8-column blocks; a
      // sequence's partials are its group's shared unit's, then its own's
      p.share_m = 16 / G;
      p.seq_batch = std::min(S, pkv::kTcMaxShareSeqs);
    }
    // decode partials: slot CTA + unit (one region per member of a shared
    // unit); any sequence of two or more chunks may be split
    p.slot_stride = (int64_t)p.n_per_group + pkv::tc_num_units(std::max(p.seq_batch, 1), p.share_m);
    p.slots = p.slot_stride * p.share_m;   // a region per member of a shared unit
    p.reduce = max_chunks > 1;
  } else {
    PKV_CHECK(simt_shape_ok(G, D), PKV_ERR_UNSUPPORTED,
              "unsupported shape: head_dim must be 32/64/128/256 and G <= 16");
    p.kind = KIND_SIMT;
    p.ps = c.num_splits ? c.num_splits : 512;
    PKV_CHECK(p.ps >= 1 && p.ps <= pkv::kSimtMaxPS, PKV_ERR_INVALID_ARGUMENT,
              "tokens per partition must be in [1, %d]", pkv::kSimtMaxPS);
    p.pmax = std::max<int>(1, (int)ceil_div(max_len, p.ps));
    PKV_CHECK(p.pmax <= 2147483647 / 2, PKV_ERR_UNSUPPORTED, "too many partitions");
    p.seq_batch = std::min(S, 65535);
    p.slots = (int64_t)std::max(p.seq_batch, 1) * p.pmax;
    p.reduce = p.pmax > 1;
  }
  p.ws_bytes = ws_layout(p, H_q, H_kv, D).total;
  *plan = p;
  return PKV_OK;
}

// Plan for a quantized pool: the tensor-core kernel when the shape allows it
// (bf16 queries, head_dim 128, G <= 8, block_size 8 or a multiple of 16, 16-byte aligned
// pools and scales), else the CUDA-core kernel (head_dim 64 / 128, G <= 16).
pkv_status plan_attention_quant(int S, int H_q, int H_kv, int D, int K, int max_len,
                                int64_t num_blocks, pkv_dtype q_dt, const pkv_kv_quant* quant,
                                const pkv_attention_config* cfg, bool aligned_ok,
                                AttnPlan* plan) {
  pkv_attention_config c = {};
  if (cfg) c = *cfg;
  PKV_CHECK(c.kernel >= 0 && c.kernel <= 2, PKV_ERR_INVALID_ARGUMENT, "bad attention config");
  PKV_CHECK(D == 64 || D == 128, PKV_ERR_UNSUPPORTED, "quantized pools need head_dim 64 or 128");
  PKV_CHECK(H_q > 0 && H_kv > 0 && H_q % H_kv == 0, PKV_ERR_INVALID_ARGUMENT,
            "num_q_heads %% num_kv_heads != 0");
  bool scales_ok = true;
  if (quant->format == PKV_KV_INT8_TOKEN && quant->k_token_scales && quant->v_token_scales)
    scales_ok = aligned(quant->k_token_scales, 16) && aligned(quant->v_token_scales, 16);
  const bool tc_ok = q_dt == PKV_BF16 && D == 128 && tc_shape_ok(H_q / H_kv, D, K, num_blocks,
                                                                  PKV_BF16) &&
                     aligned_ok && scales_ok &&
                     (quant->format != PKV_KV_BF16K_FP8V || K % 16 == 0);
  if (c.kernel == 1 || (c.kernel == 0 && tc_ok)) {
    PKV_CHECK(tc_ok, PKV_ERR_UNSUPPORTED,
              "tensor-core kernel on a one-byte pool needs bf16 queries, head_dim 128, G <= 8, "
              "block_size 8 or a multiple of 16 (a multiple of 16 with a bf16 K pool) and "
              "16-byte aligned pools and scales");
    c.kernel = 1;
    c.share_prefix = 0;   // shared-prefix groups are a bf16-pool mode
    return plan_attention(S, H_q, H_kv, D, K, max_len, num_blocks, PKV_BF16, &c, true, plan);
  }
  c.kernel = 2;
  c.share_prefix = 0;
  return plan_attention(S, H_q, H_kv, D, K, max_len, 1, q_dt, &c, false, plan);
}

pkv::Workspace carve_workspace(void* ws, const AttnPlan& p, int H_q, int H_kv, int D) {
  const WsLayout l = ws_layout(p, H_q, H_kv, D);
  uint8_t* b = static_cast<uint8_t*>(ws);
  pkv::Workspace w;
  w.meta = reinterpret_cast<int4*>(b);
  w.ml = reinterpret_cast<float2*>(b + l.ml);
  w.o = reinterpret_cast<float*>(b + l.o);
  w.pmax = p.pmax;
  return w;
}

// Shared-prefix mode: the per-group shared lengths follow the partial outputs.
int* carve_glen(void* ws, const AttnPlan& p, int H_q, int H_kv, int D) {
  return reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + ws_layout(p, H_q, H_kv, D).glen);
}

// ---- tensor-core kernel dispatch ------------------------------------------------
template <int D, int HPC, int CT, bool B8, bool SH = false>
struct TcInst {
  // stages: as many as fit in ~192 KiB (bf16) / ~203 KiB (one-byte pools)
  // of shared memory, between 2 and 8
  static constexpr int STAGE_BYTES = pkv::TcCfg<D, HPC, 2, CT>::STAGE;
  static constexpr int BUDGET = CT ? 217088 - 9216 : 196608;
  static constexpr int NS_FIT = BUDGET / STAGE_BYTES;
  static constexpr int NS = NS_FIT < 2 ? 2 : (NS_FIT > 8 ? 8 : NS_FIT);
  using C = pkv::TcCfg<D, HPC, NS, CT, B8>;
  static std::once_flag flags[kMaxDevices];
  static cudaError_t errs[kMaxDevices];
  static pkv_status launch(const pkv::TcParams& prm, int n, int groups, cudaStream_t st, int dev) {
    auto k = pkv::attn_tc_kernel<D, HPC, NS, CT, B8, SH>;
    pkv_status s = set_smem_once(k, C::SMEM, flags, errs, dev);
    if (s != PKV_OK) return s;
    PKV_CUDA(launch_pdl(k, dim3(n, groups), dim3(C::THREADS), (size_t)C::SMEM, st, prm));
    return PKV_OK;
  }
};
template <int D, int HPC, int CT, bool B8, bool SH>
std::once_flag TcInst<D, HPC, CT, B8, SH>::flags[kMaxDevices];
template <int D, int HPC, int CT, bool B8, bool SH>
cudaError_t TcInst<D, HPC, CT, B8, SH>::errs[kMaxDevices];

// ---- multi-query (prefill) kernel dispatch -----------------------------------------
template <int D, int NW>
struct PfInst {
  using C = pkv::PfCfg<D, NW>;
  static std::once_flag flags[kMaxDevices];
  static cudaError_t errs[kMaxDevices];
  static pkv_status launch(const pkv::PfParams& prm, int tiles, int H_kv, int S, cudaStream_t st,
                           int dev) {
    auto k = pkv::attn_prefill_kernel<D, NW>;
    pkv_status s = set_smem_once(k, C::SMEM, flags, errs, dev);
    if (s != PKV_OK) return s;
    PKV_CUDA(launch_pdl(k, dim3(tiles, H_kv, S), dim3(C::THREADS), (size_t)C::SMEM, st, prm));
    return PKV_OK;
  }
};
template <int D, int NW> std::once_flag PfInst<D, NW>::flags[kMaxDevices];
template <int D, int NW> cudaError_t PfInst<D, NW>::errs[kMaxDevices];


template <int D, bool SOLO>
struct X2Inst {
  using C = pkv::X2Cfg<D>;
  static std::once_flag flags[kMaxDevices];
  static cudaError_t errs[kMaxDevices];
  static pkv_status launch(const pkv::PfParams& prm, int pairs, int H_kv, int S, cudaStream_t st,
                           int dev) {
    auto k = pkv::attn_prefill_tc05x2_kernel<D, SOLO>;
    pkv_status s = set_smem_once(k, C::SMEM, flags, errs, dev);
    if (s != PKV_OK) return s;
    PKV_CUDA(launch_pdl(k, dim3(pairs, H_kv, S), dim3(C::THREADS), (size_t)C::SMEM, st, prm));
    return PKV_OK;
  }
};
template <int D, bool SOLO> std::once_flag X2Inst<D, SOLO>::flags[kMaxDevices];
template <int D, bool SOLO> cudaError_t X2Inst<D, SOLO>::errs[kMaxDevices];

// Query rows per KV head and tile: 16 per consumer warp, 1, 2 or 4 warps.
int prefill_warps(int64_t rows) { return rows <= 16 ? 1 : (rows <= 32 ? 2 : 4); }

struct PrefillPlan {
  bool tc05 = false;
  bool dec = false;        // stream-K decode kernel with several query rows per sequence
  AttnPlan ap;             // its plan
  int nw = 1;              // mma.sync kernel: consumer warps (16 rows each)
  int64_t tiles = 0;       // row tiles per (KV head, sequence)
  int nsp = 1;             // key-range splits (mma.sync kernel)
  int split_tiles = 0;     // 64-key tiles per split
  size_t ws_bytes = 0;
};

// Validates a multi-query attention call and picks the kernel, the row tiles
// and, for the mma.sync kernel, the key-range split: when the grid would be
// under four CTAs per SM and contexts span more than 8 key tiles, every CTA
// takes 8 tiles (512 keys) and the partials are merged by the split-K reduce.
pkv_status plan_prefill(int num_seqs, int num_tokens, int max_query_len, int max_context_len,
                        int H_q, int H_kv, int D, int K, int64_t num_blocks, float scale,
                        pkv_dtype dtype, const pkv_attention_config* config, PrefillPlan* out) {
  pkv_attention_config cfg = {};
  if (config) cfg = *config;
  bool reserved_zero = true;
  for (int r : cfg.reserved) reserved_zero = reserved_zero && r == 0;
  PKV_CHECK(reserved_zero && cfg.kernel >= 0 && cfg.kernel <= 3 && cfg.num_splits >= 0,
            PKV_ERR_INVALID_ARGUMENT,
            "prefill config: kernel 0 .. 3; num_splits >= 0; reserved fields 0");
  PKV_CHECK(num_seqs >= 0 && num_tokens >= 0 && max_query_len >= 0 && max_context_len >= 0 &&
                num_blocks >= 1 && K >= 1 && H_q >= 1 && H_kv >= 1 && D >= 1 && dtype_ok(dtype),
            PKV_ERR_INVALID_ARGUMENT, "bad prefill sizes");
  PKV_CHECK(H_q % H_kv == 0, PKV_ERR_INVALID_ARGUMENT,
            "num_q_heads must be a multiple of num_kv_heads");
  PKV_CHECK(max_query_len <= max_context_len, PKV_ERR_INVALID_ARGUMENT,
            "max_query_len above max_context_len");
  PKV_CHECK(std::isfinite(scale), PKV_ERR_INVALID_ARGUMENT, "scale must be finite");
  PKV_CHECK(dtype == PKV_BF16 && (D == 64 || D == 128) && (K % 16 == 0 || K == 8),
            PKV_ERR_UNSUPPORTED,
            "prefill kernel needs bf16, head_dim 64 or 128, block_size 8 or a multiple of 16");
  PKV_CHECK(num_blocks <= ((int64_t(1) << 31) - 64) / K, PKV_ERR_UNSUPPORTED,
            "pool too large for 32-bit tile rows");
  PKV_CHECK(num_seqs <= 65535 && H_kv <= 65535, PKV_ERR_UNSUPPORTED,
            "at most 65535 sequences and KV heads per call");
  // (the tcgen05 kernel folds a positive scale into its exponent and takes
  // no key-range split)
  PKV_CHECK(cfg.kernel != 1 || (scale > 0.f && cfg.num_splits <= 1), PKV_ERR_UNSUPPORTED,
            "the tcgen05 prefill kernel needs scale > 0 and no key-range split");
  PrefillPlan p;
  const int64_t rows = (int64_t)max_query_len * (H_q / H_kv);
  // up to 8 query rows per KV head: the stream-K decode kernel, queries as the
  // 8 score columns of its tensor-core tiles
  const bool dec_ok = rows <= 8 && num_seqs <= pkv::kTcMaxSeqs &&
                      (int64_t)num_tokens * H_q < (int64_t(1) << 31) &&
                      tc_shape_ok((int)std::max<int64_t>(rows, 1), D, K, num_blocks, dtype);
  PKV_CHECK(cfg.kernel != 3 || (dec_ok && cfg.num_splits == 0), PKV_ERR_UNSUPPORTED,
            "kernel 3 needs at most 8 query rows per KV head (max_query_len x G), at most "
            "2048 sequences, a tensor-core decode shape, and no key-range split");
  if (cfg.kernel == 3 || (cfg.kernel == 0 && cfg.num_splits == 0 && dec_ok)) {
    pkv_attention_config dc = {};
    dc.kernel = 1;
    pkv_status st = plan_attention(std::max(num_seqs, 1), H_q, H_kv, D, K, max_context_len,
                                   num_blocks, dtype, &dc, true, &p.ap);
    if (st != PKV_OK) return st;
    p.dec = true;
    const size_t T = (size_t)num_tokens;
    p.ws_bytes = align256(T * sizeof(int4)) + align256(T * p.ap.pmax * H_q * sizeof(float2)) +
                 align256(T * p.ap.pmax * H_q * (size_t)D * sizeof(float));
    *out = p;
    return PKV_OK;
  }
  // tcgen05 tiles of 128 rows once a KV head has more than 64 query rows;
  // mma.sync tiles of 16 / 32 / 64 rows below that
  // tcgen05 tiles of 128 rows: above 64 rows per KV head always; from 9 rows
  // when the launch has at least one 128-row tile per SM (padding rows cost
  // tensor work only, and these launches are bandwidth-bound); below that the
  // mma.sync kernel, which can split the key range over more CTAs
  bool tc05_auto = cfg.kernel == 0 && cfg.num_splits <= 1 && rows > 8 && scale > 0.f;
  if (tc05_auto && rows <= 64) {
    int dev = 0, sms = 0;
    pkv_status st = device_facts(&dev, &sms);
    if (st != PKV_OK) return st;
    tc05_auto = (int64_t)H_kv * std::max(num_seqs, 1) >= sms;
  }
  p.tc05 = cfg.kernel == 1 || tc05_auto;
  p.nw = prefill_warps(rows);
  p.tiles = std::max<int64_t>(1, ceil_div(rows, p.tc05 ? pkv::kT5Rows : 16 * p.nw));
  const int64_t max_tiles = std::max<int64_t>(1, ceil_div(max_context_len, pkv::kPfBN));
  if (!p.tc05) {
    if (cfg.num_splits > 0) {
      const int64_t want = std::min<int64_t>(cfg.num_splits, max_tiles);
      p.split_tiles = (int)ceil_div(max_tiles, want);
      p.nsp = (int)ceil_div(max_tiles, p.split_tiles);
    } else if (max_tiles > 8) {
      int dev = 0, sms = 0;
      pkv_status st = device_facts(&dev, &sms);
      if (st != PKV_OK) return st;
      if (p.tiles * H_kv * std::max(num_seqs, 1) < 4LL * sms) {
        p.split_tiles = 8;
        p.nsp = (int)ceil_div(max_tiles, 8);
      }
    }
  }
  // two 128-row tiles per CTA once a KV head has more than one
  PKV_CHECK(p.tiles * p.nsp <= 2147483647, PKV_ERR_UNSUPPORTED, "too many query rows");
  if (p.nsp > 1) {
    const size_t T = (size_t)num_tokens;
    p.ws_bytes = align256(T * sizeof(int4)) + align256(T * p.nsp * H_q * sizeof(float2)) +
                 align256(T * p.nsp * H_q * (size_t)D * sizeof(float));
  }
  *out = p;
  return PKV_OK;
}

template <int D, int CT, bool B8, bool SH = false>
pkv_status launch_tc_hpc(int hpc, const pkv::TcParams& prm, int n, int groups, cudaStream_t st,
                         int dev) {
  switch (hpc) {
    case 8: return TcInst<D, 8, CT, B8, SH>::launch(prm, n, groups, st, dev);
    case 4: return TcInst<D, 4, CT, B8, SH>::launch(prm, n, groups, st, dev);
    case 2: return TcInst<D, 2, CT, B8, SH>::launch(prm, n, groups, st, dev);
    default: return TcInst<D, 1, CT, B8, SH>::launch(prm, n, groups, st, dev);
  }
}

// 8-token blocks take the kernel's B8 layout; block sizes that are multiples
// of 16 the plain one (tensor maps from encode_pool_map_heads for both).
// Shared-prefix groups (prm.share_m > 1) exist for bf16 pools only.
template <int D, int CT>
pkv_status launch_tc_d(int hpc, int block_size, const pkv::TcParams& prm, int n, int groups,
                       cudaStream_t st, int dev) {
  if constexpr (CT == 3) {
    return launch_tc_hpc<D, CT, false>(hpc, prm, n, groups, st, dev);   // 16-row tiles only
  }
  if constexpr (CT == 0) {
    if (prm.share_m > 1)
      return block_size < pkv::kTile
                 ? launch_tc_hpc<D, CT, true, true>(hpc, prm, n, groups, st, dev)
                 : launch_tc_hpc<D, CT, false, true>(hpc, prm, n, groups, st, dev);
  }
  if constexpr (CT != 3) {
    return block_size < pkv::kTile ? launch_tc_hpc<D, CT, true>(hpc, prm, n, groups, st, dev)
                                   : launch_tc_hpc<D, CT, false>(hpc, prm, n, groups, st, dev);
  }
}

// Tensor map over a pool seen as [rows = num_blocks * K][H_kv][D] for the
// multi-query kernels: boxes of 128 bytes x 1 head x min(K, 16) rows (64 bf16
// columns, or a full 128-column row of one-byte codes), 128-byte swizzle.
pkv_status encode_pool_map(CUtensorMap* map, const void* pool, int64_t num_blocks, int K, int H_kv,
                           int D, bool one_byte = false) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  pkv_status st = get_encode(&enc);
  if (st != PKV_OK) return st;
  const cuuint64_t eb = one_byte ? 1 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H_kv, (cuuint64_t)(num_blocks * K)};
  cuuint64_t strides[2] = {(cuuint64_t)D * eb, (cuuint64_t)H_kv * D * eb};
  // one tile of 16 rows, or (8-token blocks) half a tile: a box never
  // crosses a block boundary
  cuuint32_t box[3] = {one_byte ? 128u : 64u, 1, (cuuint32_t)std::min(K, pkv::kTile)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, one_byte ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   3, const_cast<void*>(pool), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  PKV_CHECK(r == CUDA_SUCCESS, PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return PKV_OK;
}

// Tensor map over a pool for the decode kernel: dimensions (128-byte column,
// row = num_blocks * K, column group, KV head) with byte strides (row
// H_kv * D * eb, group 128, head D * eb), boxes of 128 bytes x min(K, 16)
// rows x all column groups x hpc heads, 128-byte swizzle.  A box is hpc * D
// * eb contiguous bytes of each of its rows and never crosses a block.
pkv_status encode_pool_map_heads(CUtensorMap* map, const void* pool, int64_t num_blocks, int K,
                                 int H_kv, int D, int hpc, bool one_byte) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  pkv_status st = get_encode(&enc);
  if (st != PKV_OK) return st;
  const cuuint64_t eb = one_byte ? 1 : 2;
  const cuuint64_t c0 = 128 / eb;                 // elements of a 128-byte column
  const cuuint64_t nh = (cuuint64_t)D * eb / 128; // column groups of a head row
  cuuint64_t dims[4] = {c0, (cuuint64_t)(num_blocks * K), nh, (cuuint64_t)H_kv};
  cuuint64_t strides[3] = {(cuuint64_t)H_kv * D * eb, 128, (cuuint64_t)D * eb};
  cuuint32_t box[4] = {(cuuint32_t)c0, (cuuint32_t)std::min(K, pkv::kTile), (cuuint32_t)nh,
                       (cuuint32_t)hpc};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, one_byte ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   4, const_cast<void*>(pool), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  PKV_CHECK(r == CUDA_SUCCESS, PKV_ERR_CUDA, "cuTensorMapEncodeTiled (heads) failed (%d)", (int)r);
  return PKV_OK;
}

// ---- CUDA-core kernel dispatch --------------------------------------------------
struct SimtArgs {
  const int32_t* bt;
  int maxB;
  const int32_t* lens;
  int max_len, S, H_q, H_kv, K;
  int64_t nb;
  float sl;
  pkv::Workspace ws;
  int ps, pmax;
};

template <typename T, typename KV, int D, int GMAX>
pkv_status launch_simt_t(const void* q, KV kv, void* out, const SimtArgs& a, cudaStream_t st) {
  PKV_CUDA(launch_pdl(pkv::attn_simt_kernel<T, KV, D, GMAX>, dim3(a.pmax, a.H_kv, a.S),
                      dim3(pkv::kSimtThreads), 0, st, static_cast<const T*>(q), kv, a.bt, a.maxB,
                      a.lens, a.max_len, a.H_q, a.H_kv, a.H_q / a.H_kv, a.K, (long long)a.nb,
                      a.sl, static_cast<T*>(out), a.ws, a.ps));
  return PKV_OK;
}

template <typename T, typename KV, int D>
pkv_status launch_simt_d(int G, const void* q, KV kv, void* out, const SimtArgs& a,
                         cudaStream_t st) {
  if (G <= 2) return launch_simt_t<T, KV, D, 2>(q, kv, out, a, st);
  if (G <= 8) return launch_simt_t<T, KV, D, 8>(q, kv, out, a, st);
  return launch_simt_t<T, KV, D, 16>(q, kv, out, a, st);
}

template <typename T, typename KV>
pkv_status launch_simt(int D, const void* q, KV kv, void* out, const SimtArgs& a,
                       cudaStream_t st) {
  const int G = a.H_q / a.H_kv;
  switch (D) {
    case 32: return launch_simt_d<T, KV, 32>(G, q, kv, out, a, st);
    case 64: return launch_simt_d<T, KV, 64>(G, q, kv, out, a, st);
    case 128: return launch_simt_d<T, KV, 128>(G, q, kv, out, a, st);
    default: return launch_simt_d<T, KV, 256>(G, q, kv, out, a, st);
  }
}

// Quantized pools: head_dim 64 or 128 only (fewer instantiations).
template <typename T, typename KV>
pkv_status launch_simt_q(int D, const void* q, KV kv, void* out, const SimtArgs& a,
                         cudaStream_t st) {
  const int G = a.H_q / a.H_kv;
  if (D == 64) return launch_simt_d<T, KV, 64>(G, q, kv, out, a, st);
  return launch_simt_d<T, KV, 128>(G, q, kv, out, a, st);
}

template <typename T>
pkv_status launch_simt_typed(const pkv_kv_quant* quant, int D, const void* q, const void* kc,
                             const void* vc, void* out, const SimtArgs& a, cudaStream_t st) {
  if (quant == nullptr)
    return launch_simt<T>(D, q, pkv::KvPlain<T>{static_cast<const T*>(kc),
                                                 static_cast<const T*>(vc)}, out, a, st);
  if (quant->format == PKV_KV_FP8_E4M3)
    return launch_simt_q<T>(D, q, pkv::KvFp8{static_cast<const uint8_t*>(kc),
                                              static_cast<const uint8_t*>(vc), quant->k_scale,
                                              quant->v_scale}, out, a, st);
  if (quant->format == PKV_KV_BF16K_FP8V)
    return launch_simt_q<T>(D, q, pkv::KvBf16Fp8{static_cast<const __nv_bfloat16*>(kc),
                                                  static_cast<const uint8_t*>(vc),
                                                  quant->v_scale}, out, a, st);
  return launch_simt_q<T>(D, q, pkv::KvInt8{static_cast<const int8_t*>(kc),
                                             static_cast<const int8_t*>(vc),
                                             quant->k_token_scales, quant->v_token_scales},
                          out, a, st);
}

pkv_status launch_simt_any(pkv_dtype dt, const pkv_kv_quant* quant, int D, const void* q,
                           const void* kc, const void* vc, void* out, const SimtArgs& a,
                           cudaStream_t st) {
  return dt == PKV_BF16 ? launch_simt_typed<__nv_bfloat16>(quant, D, q, kc, vc, out, a, st)
                        : launch_simt_typed<float>(quant, D, q, kc, vc, out, a, st);
}

// ---- split-K reduce dispatch -----------------------------------------------------
template <typename T>
pkv_status launch_reduce(int D, pkv::Workspace ws, int S, int H_q, void* out, cudaStream_t st) {
  const int64_t pairs = (int64_t)S * H_q;
  const dim3 grid((unsigned)ceil_div(pairs, pkv::kReduceWarps));
  const dim3 block(pkv::kReduceWarps * 32);
  T* o = static_cast<T*>(out);
  switch (D) {
    case 32: PKV_CUDA(launch_pdl(pkv::attn_reduce_kernel<T, 32>, grid, block, 0, st, ws, S, H_q, o)); break;
    case 64: PKV_CUDA(launch_pdl(pkv::attn_reduce_kernel<T, 64>, grid, block, 0, st, ws, S, H_q, o)); break;
    case 128: PKV_CUDA(launch_pdl(pkv::attn_reduce_kernel<T, 128>, grid, block, 0, st, ws, S, H_q, o)); break;
    default: PKV_CUDA(launch_pdl(pkv::attn_reduce_kernel<T, 256>, grid, block, 0, st, ws, S, H_q, o)); break;
  }
  return PKV_OK;
}

// Widest vector (16/8/4/2/1 bytes) that divides the row and every base pointer.
int vec_width(int64_t row_bytes, std::initializer_list<const void*> ptrs) {
  for (int w : {16, 8, 4, 2, 1}) {
    if (row_bytes % w) continue;
    bool ok = true;
    for (const void* p : ptrs) ok = ok && aligned(p, w);
    if (ok) return w;
  }
  return 0;
}

// Moves whole blocks of `blk` bytes from the source pools to the destination
// pools for every (src, dst) pair; src_v / dst_v null means one tensor.
pkv_status move_blocks(const void* src_k, const void* src_v, int64_t src_nb, void* dst_k,
                       void* dst_v, int64_t dst_nb, const int64_t* pairs, int64_t num_pairs,
                       int64_t blk, cudaStream_t st) {
  PKV_CHECK(num_pairs <= 2147483647, PKV_ERR_UNSUPPORTED, "too many pairs");
  const bool two = src_v != nullptr;
  const int vw = two ? vec_width(blk, {src_k, src_v, dst_k, dst_v}) : vec_width(blk, {src_k, dst_k});
  PKV_CHECK(vw > 0, PKV_ERR_INVALID_ARGUMENT, "misaligned pools");
  constexpr int threads = 256, unroll = 4;
  const int64_t chunks = ceil_div(blk / vw, threads * unroll);
  PKV_CHECK(chunks <= 65535, PKV_ERR_UNSUPPORTED, "block too large");
  dim3 grid((unsigned)num_pairs, (unsigned)chunks, two ? 2 : 1);
  auto* sk = static_cast<const uint8_t*>(src_k);
  auto* sv = static_cast<const uint8_t*>(src_v);
  auto* dk = static_cast<uint8_t*>(dst_k);
  auto* dv = static_cast<uint8_t*>(dst_v);
#define PKV_MOVE(W)                                                                           \
  PKV_CUDA(launch_pdl(pkv::block_move_kernel<W, unroll>, grid, dim3(threads), 0, st, sk, sv, \
                      dk, dv, pairs, src_nb, dst_nb, blk))
  switch (vw) {
    case 16: PKV_MOVE(16); break;
    case 8: PKV_MOVE(8); break;
    case 4: PKV_MOVE(4); break;
    case 2: PKV_MOVE(2); break;
    default: PKV_MOVE(1); break;
  }
#undef PKV_MOVE
  return PKV_OK;
}

// Copy-on-write: blocks move within one pool.
pkv_status copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs, int64_t num_pairs,
                       int64_t num_blocks, int64_t blk, cudaStream_t st) {
  return move_blocks(k_cache, v_cache, num_blocks, k_cache, v_cache, num_blocks, pairs, num_pairs,
                     blk, st);
}

// The address kernels use for a caller's buffer: device memory of the current
// device as it is, page-locked host memory through its device mapping.
// Pageable host memory and other devices' memory are refused.
pkv_status device_view(const void* p, const char* what, const void** out) {
  cudaPointerAttributes a{};
  const cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(PKV_ERR_INVALID_ARGUMENT, "%s: not a CUDA-visible pointer", what);
  }
  int dev = -1;
  PKV_CUDA(cudaGetDevice(&dev));
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      PKV_CHECK(a.device == dev, PKV_ERR_INVALID_ARGUMENT, "%s: memory of another device", what);
      *out = a.devicePointer;
      return PKV_OK;
    case cudaMemoryTypeHost:
      PKV_CHECK(a.devicePointer != nullptr, PKV_ERR_INVALID_ARGUMENT,
                "%s: page-locked host memory not mapped for this device", what);
      *out = a.devicePointer;
      return PKV_OK;
    default:
      return fail(PKV_ERR_INVALID_ARGUMENT,
                  "%s: pageable host memory (pin it: cudaHostAlloc / cudaHostRegister)", what);
  }
}

// Validates a quantized-pool description (token scales required for INT8).
pkv_status check_quant(const pkv_kv_quant* q, bool need_token_scales) {
  PKV_CHECK(q != nullptr, PKV_ERR_INVALID_ARGUMENT, "null quant description");
  PKV_CHECK(q->format == PKV_KV_FP8_E4M3 || q->format == PKV_KV_INT8_TOKEN ||
                q->format == PKV_KV_BF16K_FP8V,
            PKV_ERR_INVALID_ARGUMENT, "quant format must be FP8_E4M3, INT8_TOKEN or BF16K_FP8V");
  if (q->format == PKV_KV_FP8_E4M3) {
    PKV_CHECK(std::isfinite(q->k_scale) && std::isfinite(q->v_scale) && q->k_scale > 0.f &&
                  q->v_scale > 0.f,
              PKV_ERR_INVALID_ARGUMENT, "FP8 scales must be finite and > 0");
  } else if (q->format == PKV_KV_BF16K_FP8V) {
    PKV_CHECK(std::isfinite(q->v_scale) && q->v_scale > 0.f, PKV_ERR_INVALID_ARGUMENT,
              "the FP8 V scale must be finite and > 0");
  } else if (need_token_scales) {
    PKV_CHECK(q->k_token_scales && q->v_token_scales, PKV_ERR_INVALID_ARGUMENT,
              "INT8 pools need per-token scale arrays");
    PKV_CHECK(aligned(q->k_token_scales, 4) && aligned(q->v_token_scales, 4),
              PKV_ERR_INVALID_ARGUMENT, "misaligned token scales");
  }
  return PKV_OK;
}

// ---- fixed scratch for pkv_attention_decode_noalloc ---------------------------
// In host code this name is only a host-side stand-in for the array; the
// device address is looked up per device with cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

struct NoAllocScratch {
  std::mutex mu;
  void* ptr = nullptr;   // set only once a lookup has succeeded
};
NoAllocScratch g_noalloc[kMaxDevices];

// Device address of this device's copy of the scratch array, looked up with
// that device current.  Only a successful lookup is kept: a failed one (for
// instance the module could not be loaded because the device's memory was
// full) returns its error and the next call tries again.
pkv_status noalloc_scratch(void** ptr) {
  int dev = 0;
  PKV_CUDA(cudaGetDevice(&dev));
  PKV_CHECK(dev >= 0 && dev < kMaxDevices, PKV_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
  NoAllocScratch& sc = g_noalloc[dev];
  std::lock_guard<std::mutex> lock(sc.mu);
  if (sc.ptr == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return fail(PKV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    }
    sc.ptr = p;
  }
  *ptr = sc.ptr;
  return PKV_OK;
}

}  // namespace

// =============================================================================
// C ABI
// =============================================================================
extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARGUMENT: return "PKV_ERR_INVALID_ARGUMENT";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "PKV_ERR_WORKSPACE_TOO_SMALL";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_DEVICE_CHECK: return "PKV_ERR_DEVICE_CHECK";
  }
  return "PKV_UNKNOWN_STATUS";
}

const char* pkv_last_error_message(void) { return g_last_msg.c_str(); }

int32_t pkv_version(void) { return (1 << 16) | 0; }

pkv_status pkv_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* positions, int32_t num_seqs, int32_t block_size,
                            int64_t num_blocks, int64_t* slot_mapping, void* stream) {
  PKV_CHECK(num_seqs >= 0 && max_blocks_per_seq >= 1 && block_size >= 1 && num_blocks >= 1,
            PKV_ERR_INVALID_ARGUMENT, "bad slot-mapping sizes");
  if (num_seqs == 0) return PKV_OK;
  PKV_CHECK(block_tables && positions && slot_mapping, PKV_ERR_INVALID_ARGUMENT, "null pointer");
  PKV_CHECK(num_blocks <= INT64_MAX / block_size, PKV_ERR_INVALID_ARGUMENT, "pool too large");
  const int threads = 256;
  PKV_CUDA(launch_pdl(pkv::slot_mapping_kernel, dim3((num_seqs + threads - 1) / threads),
                      dim3(threads), 0, as_stream(stream), block_tables, max_blocks_per_seq,
                      positions, num_seqs, block_size, log2_exact(block_size), num_blocks,
                      slot_mapping));
  return PKV_OK;
}

pkv_status pkv_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                        int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_blocks,
                        int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                        pkv_dtype dtype, void* stream) {
  PKV_CHECK(num_tokens >= 0 && num_blocks >= 1 && block_size >= 1 && num_kv_heads >= 1 &&
                head_dim >= 1 && dtype_ok(dtype),
            PKV_ERR_INVALID_ARGUMENT, "bad kv_write sizes");
  if (num_tokens == 0) return PKV_OK;
  PKV_CHECK(k && v && slot_mapping && k_cache && v_cache, PKV_ERR_INVALID_ARGUMENT, "null pointer");
  PKV_CHECK(num_tokens <= 2147483647, PKV_ERR_UNSUPPORTED, "too many tokens");
  const int64_t row = (int64_t)num_kv_heads * head_dim * elem_bytes(dtype);
  const int vw = vec_width(row, {k, v, k_cache, v_cache});
  PKV_CHECK(vw >= 2, PKV_ERR_INVALID_ARGUMENT, "misaligned kv_write buffers");
  const int threads = 128;
  const int64_t nvec = row / vw;
  const int64_t chunks = ceil_div(nvec, threads);
  PKV_CHECK(chunks <= 65535, PKV_ERR_UNSUPPORTED, "token row too wide");
  dim3 grid((unsigned)num_tokens, (unsigned)chunks, 2);
  const int64_t slots = num_blocks * block_size;
  auto* kb = static_cast<const uint8_t*>(k);
  auto* vb = static_cast<const uint8_t*>(v);
  auto* kc = static_cast<uint8_t*>(k_cache);
  auto* vc = static_cast<uint8_t*>(v_cache);
  cudaStream_t st = as_stream(stream);
  switch (vw) {
    case 16: PKV_CUDA(launch_pdl(pkv::kv_write_kernel<16>, grid, dim3(threads), 0, st, kb, vb, slot_mapping, kc, vc, slots, row)); break;
    case 8: PKV_CUDA(launch_pdl(pkv::kv_write_kernel<8>, grid, dim3(threads), 0, st, kb, vb, slot_mapping, kc, vc, slots, row)); break;
    case 4: PKV_CUDA(launch_pdl(pkv::kv_write_kernel<4>, grid, dim3(threads), 0, st, kb, vb, slot_mapping, kc, vc, slots, row)); break;
    default: PKV_CUDA(launch_pdl(pkv::kv_write_kernel<2>, grid, dim3(threads), 0, st, kb, vb, slot_mapping, kc, vc, slots, row)); break;
  }
  return PKV_OK;
}

pkv_status pkv_kv_append(const void* k, const void* v, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* positions, int32_t num_tokens,
                         void* k_cache, void* v_cache, int64_t num_blocks, int32_t block_size,
                         int32_t num_kv_heads, int32_t head_dim, pkv_dtype dtype,
                         int64_t* slot_mapping_out, void* stream) {
  PKV_CHECK(num_tokens >= 0 && max_blocks_per_seq >= 1 && num_blocks >= 1 && block_size >= 1 &&
                num_kv_heads >= 1 && head_dim >= 1 && dtype_ok(dtype),
            PKV_ERR_INVALID_ARGUMENT, "bad kv_append sizes");
  if (num_tokens == 0) return PKV_OK;
  PKV_CHECK(k && v && block_tables && positions && k_cache && v_cache, PKV_ERR_INVALID_ARGUMENT,
            "null pointer");
  PKV_CHECK(num_blocks <= INT64_MAX / block_size, PKV_ERR_INVALID_ARGUMENT, "pool too large");
  const int64_t row = (int64_t)num_kv_heads * head_dim * elem_bytes(dtype);
  const int vw = vec_width(row, {k, v, k_cache, v_cache});
  PKV_CHECK(vw >= 2, PKV_ERR_INVALID_ARGUMENT, "misaligned kv_append buffers");
  const int threads = 128;
  const int64_t chunks = ceil_div(row / vw, threads);
  PKV_CHECK(chunks <= 65535, PKV_ERR_UNSUPPORTED, "token row too wide");
  dim3 grid((unsigned)num_tokens, (unsigned)chunks, 2);
  auto* kb = static_cast<const uint8_t*>(k);
  auto* vb = static_cast<const uint8_t*>(v);
  auto* kc = static_cast<uint8_t*>(k_cache);
  auto* vc = static_cast<uint8_t*>(v_cache);
  const int l2 = log2_exact(block_size);
  cudaStream_t st = as_stream(stream);
  switch (vw) {
    case 16: PKV_CUDA(launch_pdl(pkv::kv_append_kernel<16>, grid, dim3(threads), 0, st, kb, vb, block_tables, max_blocks_per_seq, positions, block_size, l2, num_blocks, kc, vc, row, slot_mapping_out)); break;
    case 8: PKV_CUDA(launch_pdl(pkv::kv_append_kernel<8>, grid, dim3(threads), 0, st, kb, vb, block_tables, max_blocks_per_seq, positions, block_size, l2, num_blocks, kc, vc, row, slot_mapping_out)); break;
    case 4: PKV_CUDA(launch_pdl(pkv::kv_append_kernel<4>, grid, dim3(threads), 0, st, kb, vb, block_tables, max_blocks_per_seq, positions, block_size, l2, num_blocks, kc, vc, row, slot_mapping_out)); break;
    default: PKV_CUDA(launch_pdl(pkv::kv_append_kernel<2>, grid, dim3(threads), 0, st, kb, vb, block_tables, max_blocks_per_seq, positions, block_size, l2, num_blocks, kc, vc, row, slot_mapping_out)); break;
  }
  return PKV_OK;
}

pkv_status pkv_selftest_wait_timeout(int64_t limit_cycles, void* stream) {
  PKV_CHECK(limit_cycles >= 1 && limit_cycles <= (int64_t(1) << 31), PKV_ERR_INVALID_ARGUMENT,
            "limit_cycles must be in [1, 2^31]");
  pkv::selftest_wait_timeout_kernel<<<1, 32, 0, as_stream(stream)>>>((long long)limit_cycles);
  PKV_CUDA(cudaGetLastError());
  return PKV_OK;
}

pkv_status pkv_kv_block_copy(void* k_cache, void* v_cache, const int64_t* src_dst_pairs,
                             int64_t num_pairs, int64_t num_blocks, int32_t block_size,
                             int32_t num_kv_heads, int32_t head_dim, pkv_dtype dtype,
                             void* stream) {
  PKV_CHECK(num_pairs >= 0 && num_blocks >= 1 && block_size >= 1 && num_kv_heads >= 1 &&
                head_dim >= 1 && dtype_ok(dtype),
            PKV_ERR_INVALID_ARGUMENT, "bad block-copy sizes");
  if (num_pairs == 0) return PKV_OK;
  PKV_CHECK(k_cache && v_cache && src_dst_pairs, PKV_ERR_INVALID_ARGUMENT, "null pointer");
  const int64_t blk = (int64_t)block_size * num_kv_heads * head_dim * elem_bytes(dtype);
  return copy_blocks(k_cache, v_cache, src_dst_pairs, num_pairs, num_blocks, blk,
                     as_stream(stream));
}

pkv_status pkv_kv_block_swap(const void* src_k, const void* src_v, int64_t src_num_blocks,
                             void* dst_k, void* dst_v, int64_t dst_num_blocks, int64_t block_bytes,
                             const int64_t* pairs, int64_t num_pairs, void* stream) {
  PKV_CHECK(num_pairs >= 0 && src_num_blocks >= 1 && dst_num_blocks >= 1 && block_bytes >= 1,
            PKV_ERR_INVALID_ARGUMENT, "bad block-swap sizes");
  PKV_CHECK((src_v == nullptr) == (dst_v == nullptr), PKV_ERR_INVALID_ARGUMENT,
            "src_v and dst_v must both be given or both be NULL");
  PKV_CHECK(src_num_blocks <= INT64_MAX / block_bytes && dst_num_blocks <= INT64_MAX / block_bytes,
            PKV_ERR_INVALID_ARGUMENT, "pool too large");
  if (num_pairs == 0) return PKV_OK;
  PKV_CHECK(src_k && dst_k && pairs, PKV_ERR_INVALID_ARGUMENT, "null pointer");
  PKV_CHECK(aligned(pairs, 8), PKV_ERR_INVALID_ARGUMENT, "misaligned pairs");
  const void *sk = nullptr, *sv = nullptr, *dk = nullptr, *dv = nullptr, *pr = nullptr;
  pkv_status st = device_view(src_k, "src_k", &sk);
  if (st == PKV_OK) st = device_view(dst_k, "dst_k", &dk);
  if (st == PKV_OK && src_v) st = device_view(src_v, "src_v", &sv);
  if (st == PKV_OK && dst_v) st = device_view(dst_v, "dst_v", &dv);
  if (st == PKV_OK) st = device_view(pairs, "pairs", &pr);
  if (st != PKV_OK) return st;
  return move_blocks(sk, sv, src_num_blocks, const_cast<void*>(dk), const_cast<void*>(dv),
                     dst_num_blocks, static_cast<const int64_t*>(pr), num_pairs, block_bytes,
                     as_stream(stream));
}

pkv_status pkv_kv_append_quant(const void* k, const void* v, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* positions,
                               int32_t num_tokens, void* k_cache, void* v_cache,
                               int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                               int32_t head_dim, pkv_dtype in_dtype, const pkv_kv_quant* quant,
                               int64_t* slot_mapping_out, void* stream) {
  PKV_CHECK(num_tokens >= 0 && max_blocks_per_seq >= 1 && num_blocks >= 1 && block_size >= 1 &&
                num_kv_heads >= 1 && head_dim >= 1 && dtype_ok(in_dtype),
            PKV_ERR_INVALID_ARGUMENT, "bad kv_append_quant sizes");
  pkv_status st = check_quant(quant, true);
  if (st != PKV_OK) return st;
  if (num_tokens == 0) return PKV_OK;
  PKV_CHECK(k && v && block_tables && positions && k_cache && v_cache, PKV_ERR_INVALID_ARGUMENT,
            "null pointer");
  PKV_CHECK(num_blocks <= INT64_MAX / block_size, PKV_ERR_INVALID_ARGUMENT, "pool too large");
  PKV_CHECK(aligned(k, elem_bytes(in_dtype)) && aligned(v, elem_bytes(in_dtype)),
            PKV_ERR_INVALID_ARGUMENT, "misaligned k/v");
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  const int l2 = log2_exact(block_size);
  dim3 grid((unsigned)num_tokens, 2);
  dim3 block(pkv::kQuantThreads);
  cudaStream_t strm = as_stream(stream);
  auto* kc = static_cast<uint8_t*>(k_cache);
  auto* vc = static_cast<uint8_t*>(v_cache);
  const float ks = quant->k_scale, vs = quant->v_scale;
  float* kts = quant->k_token_scales;
  float* vts = quant->v_token_scales;
#define PKV_LAUNCH_AQ(TIN, FMT)                                                               \
  PKV_CUDA(launch_pdl(pkv::kv_append_quant_kernel<TIN, FMT>, grid, block, 0, strm,            \
                      static_cast<const TIN*>(k), static_cast<const TIN*>(v), block_tables,   \
                      max_blocks_per_seq, positions, block_size, l2, num_blocks, kc, vc, row, \
                      ks, vs, kts, vts, slot_mapping_out))
  if (quant->format == PKV_KV_FP8_E4M3) {
    if (in_dtype == PKV_BF16) PKV_LAUNCH_AQ(__nv_bfloat16, 1); else PKV_LAUNCH_AQ(float, 1);
  } else if (quant->format == PKV_KV_BF16K_FP8V) {
    PKV_CHECK(aligned(k_cache, 2), PKV_ERR_INVALID_ARGUMENT, "misaligned bf16 K pool");
    if (in_dtype == PKV_BF16) PKV_LAUNCH_AQ(__nv_bfloat16, 3); else PKV_LAUNCH_AQ(float, 3);
  } else {
    if (in_dtype == PKV_BF16) PKV_LAUNCH_AQ(__nv_bfloat16, 2); else PKV_LAUNCH_AQ(float, 2);
  }
#undef PKV_LAUNCH_AQ
  return PKV_OK;
}

pkv_status pkv_kv_block_copy_quant(void* k_cache, void* v_cache, const int64_t* src_dst_pairs,
                                   int64_t num_pairs, int64_t num_blocks, int32_t block_size,
                                   int32_t num_kv_heads, int32_t head_dim,
                                   const pkv_kv_quant* quant, void* stream) {
  PKV_CHECK(num_pairs >= 0 && num_blocks >= 1 && block_size >= 1 && num_kv_heads >= 1 &&
                head_dim >= 1,
            PKV_ERR_INVALID_ARGUMENT, "bad block-copy sizes");
  pkv_status st = check_quant(quant, true);
  if (st != PKV_OK) return st;
  if (num_pairs == 0) return PKV_OK;
  PKV_CHECK(k_cache && v_cache && src_dst_pairs, PKV_ERR_INVALID_ARGUMENT, "null pointer");
  const int64_t blk = (int64_t)block_size * num_kv_heads * head_dim;
  cudaStream_t strm = as_stream(stream);
  if (quant->format == PKV_KV_BF16K_FP8V) {
    // two pools of different block sizes: K (2 bytes per element), then V
    st = move_blocks(k_cache, nullptr, num_blocks, k_cache, nullptr, num_blocks, src_dst_pairs,
                     num_pairs, 2 * blk, strm);
    if (st != PKV_OK) return st;
    return move_blocks(v_cache, nullptr, num_blocks, v_cache, nullptr, num_blocks,
                       src_dst_pairs, num_pairs, blk, strm);
  }
  st = copy_blocks(k_cache, v_cache, src_dst_pairs, num_pairs, num_blocks, blk, strm);
  if (st != PKV_OK) return st;
  if (quant->format == PKV_KV_INT8_TOKEN) {
    PKV_CUDA(launch_pdl(pkv::token_scale_copy_kernel, dim3((unsigned)num_pairs), dim3(64), 0,
                        strm, quant->k_token_scales, quant->v_token_scales, src_dst_pairs,
                        num_blocks, block_size));
  }
  return PKV_OK;
}

pkv_status pkv_attention_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         int32_t block_size, int32_t max_context_len,
                                         pkv_dtype dtype, const pkv_attention_config* config,
                                         size_t* bytes) {
  PKV_CHECK(bytes != nullptr, PKV_ERR_INVALID_ARGUMENT, "null bytes pointer");
  AttnPlan plan;
  // the tensor-core plan assumes an aligned pool; a misaligned pool takes the
  // CUDA-core plan, whose workspace is never larger for the same sizes
  pkv_status st = plan_attention(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_context_len, 1, dtype, config, true, &plan);
  if (st != PKV_OK) return st;
  AttnPlan alt;
  pkv_attention_config c2 = {};
  if (config) c2 = *config;
  if (plan.kind == KIND_TC && c2.kernel == 0) {
    c2.kernel = 2;
    c2.num_splits = 0;
    if (plan_attention(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                       1, dtype, &c2, true, &alt) == PKV_OK)
      plan.ws_bytes = std::max(plan.ws_bytes, alt.ws_bytes);
  }
  *bytes = plan.ws_bytes;
  return PKV_OK;
}

pkv_status pkv_attention_launch_count(int32_t num_seqs, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                      int32_t max_context_len, pkv_dtype dtype,
                                      const pkv_attention_config* config, int32_t* launches) {
  PKV_CHECK(launches != nullptr, PKV_ERR_INVALID_ARGUMENT, "null launches pointer");
  AttnPlan plan;
  pkv_status st = plan_attention(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_context_len, 1, dtype, config, true, &plan);
  if (st != PKV_OK) return st;
  const int batches = num_seqs == 0 ? 0 : (int)ceil_div(num_seqs, plan.seq_batch);
  // partition (+ split-K reduce) (+ the table comparison of share_prefix)
  *launches = batches * (1 + (plan.reduce ? 1 : 0) + (plan.share_m > 1 ? 1 : 0));
  return PKV_OK;
}

}  // extern "C"

namespace {

pkv_status attention_impl(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* context_lens, int32_t max_context_len, int32_t num_seqs,
                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int64_t num_blocks, float scale, void* out,
                          void* workspace, size_t workspace_bytes, pkv_dtype dtype,
                          const pkv_attention_config* config, const pkv_kv_quant* quant,
                          void* stream) {
  PKV_CHECK(num_seqs >= 0 && max_blocks_per_seq >= 1 && num_blocks >= 1,
            PKV_ERR_INVALID_ARGUMENT, "bad attention sizes");
  const bool tma_aligned = aligned(k_cache, 16) && aligned(v_cache, 16);
  AttnPlan plan;
  pkv_status st = quant ? plan_attention_quant(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                               block_size, max_context_len, num_blocks, dtype,
                                               quant, config, tma_aligned, &plan)
                        : plan_attention(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                         block_size, max_context_len, num_blocks, dtype, config,
                                         tma_aligned, &plan);
  if (st != PKV_OK) return st;
  if (num_seqs == 0) return PKV_OK;
  PKV_CHECK(q && k_cache && v_cache && block_tables && context_lens && out && workspace,
            PKV_ERR_INVALID_ARGUMENT, "null pointer");
  PKV_CHECK(workspace_bytes >= plan.ws_bytes, PKV_ERR_WORKSPACE_TOO_SMALL,
            "workspace %zu bytes < %zu needed", workspace_bytes, plan.ws_bytes);
  PKV_CHECK(aligned(workspace, 256), PKV_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  const size_t eb = elem_bytes(dtype);
  const size_t pool_eb = quant ? 1 : eb;
  const size_t k_eb = quant && quant->format == PKV_KV_BF16K_FP8V ? 2 : pool_eb;
  PKV_CHECK(aligned(q, eb) && aligned(out, eb) && aligned(k_cache, k_eb) &&
                aligned(v_cache, pool_eb),
            PKV_ERR_INVALID_ARGUMENT, "misaligned q/out/pool");
  PKV_CHECK((int64_t)max_blocks_per_seq * block_size <= 2147483647, PKV_ERR_UNSUPPORTED,
            "table row too long");
  const double log2e = 1.4426950408889634;
  const float sl = (float)((double)scale * log2e);
  cudaStream_t strm = as_stream(stream);
  pkv::Workspace ws = carve_workspace(workspace, plan, num_q_heads, num_kv_heads, head_dim);
  const int D = head_dim, H_q = num_q_heads, H_kv = num_kv_heads;

  pkv::TcParams prm;
  int dev = 0;
  if (plan.kind == KIND_TC) {
    int sms;
    st = device_facts(&dev, &sms);
    if (st != PKV_OK) return st;
    memset(&prm, 0, sizeof(prm));
    // one-byte tiles for quantized pools, except the bf16 K pool of the pair
    const bool k16 = quant != nullptr && quant->format == PKV_KV_BF16K_FP8V;
    st = encode_pool_map_heads(&prm.tmap_k, k_cache, num_blocks, block_size, H_kv, D, plan.hpc,
                               quant != nullptr && !k16);
    if (st != PKV_OK) return st;
    st = encode_pool_map_heads(&prm.tmap_v, v_cache, num_blocks, block_size, H_kv, D, plan.hpc,
                               quant != nullptr);
    if (st != PKV_OK) return st;
    if (quant) {
      prm.v_scale = quant->format == PKV_KV_INT8_TOKEN ? 1.f : quant->v_scale;
      prm.k_ts = quant->k_token_scales;
      prm.v_ts = quant->v_token_scales;
    }
  }
  for (int s0 = 0; s0 < num_seqs; s0 += plan.seq_batch) {
    const int S = std::min(plan.seq_batch, num_seqs - s0);
    const uint8_t* qb = static_cast<const uint8_t*>(q) + (size_t)s0 * H_q * D * eb;
    uint8_t* ob = static_cast<uint8_t*>(out) + (size_t)s0 * H_q * D * eb;
    const int32_t* btb = block_tables + (size_t)s0 * max_blocks_per_seq;
    const int32_t* lb = context_lens + s0;
    if (plan.kind == KIND_TC) {
      prm.q = reinterpret_cast<const __nv_bfloat16*>(qb);
      prm.out = reinterpret_cast<__nv_bfloat16*>(ob);
      prm.block_tables = btb;
      prm.context_lens = lb;
      prm.ws = ws;
      prm.num_blocks = num_blocks;
      prm.max_blocks_per_seq = max_blocks_per_seq;
      prm.num_seqs = S;
      prm.max_len = max_context_len;
      prm.H_q = H_q;
      prm.G = H_q / H_kv;
      prm.block_size = block_size;
      prm.scale_log2 = sl;
      prm.share_m = plan.share_m;
      prm.slot_stride = plan.share_m > 1 ? (int)plan.slot_stride : 0;
      prm.glen = nullptr;
      if (plan.share_m > 1) {
        // the groups' shared lengths, from the table rows
        int* glen = carve_glen(workspace, plan, H_q, H_kv, D);
        const int ngroups = (int)ceil_div(S, plan.share_m);
        PKV_CUDA(launch_pdl(pkv::share_prefix_kernel,
                            dim3((unsigned)ceil_div(ngroups, pkv::kShareWarps)),
                            dim3(pkv::kShareWarps * 32), 0, strm, btb, max_blocks_per_seq, lb,
                            max_context_len, S, block_size, plan.share_m, glen));
        prm.glen = glen;
      }
      if (quant == nullptr) {
        st = D == 64 ? launch_tc_d<64, 0>(plan.hpc, block_size, prm, plan.n_per_group, plan.groups,
                                          strm, dev)
                     : launch_tc_d<128, 0>(plan.hpc, block_size, prm, plan.n_per_group,
                                           plan.groups, strm, dev);
      } else if (quant->format == PKV_KV_FP8_E4M3) {
        prm.scale_log2 = (float)((double)scale * log2e * (double)quant->k_scale);
        st = launch_tc_d<128, 1>(plan.hpc, block_size, prm, plan.n_per_group, plan.groups, strm,
                                 dev);
      } else if (quant->format == PKV_KV_BF16K_FP8V) {
        st = launch_tc_d<128, 3>(plan.hpc, block_size, prm, plan.n_per_group, plan.groups, strm,
                                 dev);
      } else {
        st = launch_tc_d<128, 2>(plan.hpc, block_size, prm, plan.n_per_group, plan.groups, strm,
                                 dev);
      }
    } else {
      const SimtArgs a{btb, max_blocks_per_seq, lb, max_context_len, S, H_q, H_kv,
                       block_size, num_blocks, sl, ws, plan.ps, plan.pmax};
      st = launch_simt_any(dtype, quant, D, qb, k_cache, v_cache, ob, a, strm);
    }
    if (st != PKV_OK) return st;
    if (plan.reduce) {
      st = dtype == PKV_BF16
               ? launch_reduce<__nv_bfloat16>(D, ws, S, H_q, ob, strm)
               : launch_reduce<float>(D, ws, S, H_q, ob, strm);
      if (st != PKV_OK) return st;
    }
  }
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, int32_t max_context_len,
                                int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                float scale, void* out, void* workspace, size_t workspace_bytes,
                                pkv_dtype dtype, const pkv_attention_config* config,
                                void* stream) {
  return attention_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                        block_size, num_blocks, scale, out, workspace, workspace_bytes, dtype,
                        config, nullptr, stream);
}

pkv_status pkv_attention_decode_quant(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t max_context_len,
                                      int32_t num_seqs, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int64_t num_blocks, float scale,
                                      void* out, void* workspace, size_t workspace_bytes,
                                      pkv_dtype q_dtype, const pkv_kv_quant* quant,
                                      const pkv_attention_config* config, void* stream) {
  pkv_status st = check_quant(quant, true);
  if (st != PKV_OK) return st;
  return attention_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                        block_size, num_blocks, scale, out, workspace, workspace_bytes, q_dtype,
                        config, quant, stream);
}

pkv_status pkv_attention_quant_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                               int32_t num_kv_heads, int32_t head_dim,
                                               int32_t block_size, int32_t max_context_len,
                                               pkv_dtype q_dtype, const pkv_kv_quant* quant,
                                               const pkv_attention_config* config,
                                               size_t* bytes) {
  PKV_CHECK(bytes != nullptr, PKV_ERR_INVALID_ARGUMENT, "null bytes pointer");
  pkv_status st = check_quant(quant, false);
  if (st != PKV_OK) return st;
  // aligned pools are assumed; a misaligned pool takes the CUDA-core plan,
  // so report the larger of the two workspaces
  AttnPlan plan;
  st = plan_attention_quant(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                            max_context_len, 1, q_dtype, quant, config, true, &plan);
  if (st != PKV_OK) return st;
  size_t need = plan.ws_bytes;
  pkv_attention_config c2 = {};
  if (config) c2 = *config;
  if (plan.kind == KIND_TC && c2.kernel == 0) {
    c2.kernel = 2;
    c2.num_splits = 0;
    AttnPlan alt;
    if (plan_attention_quant(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                             max_context_len, 1, q_dtype, quant, &c2, true, &alt) == PKV_OK)
      need = std::max(need, alt.ws_bytes);
  }
  *bytes = need;
  return PKV_OK;
}

pkv_status pkv_attention_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t max_context_len,
                                        int32_t num_seqs, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t block_size, int64_t num_blocks, float scale,
                                        void* out, pkv_dtype dtype,
                                        const pkv_attention_config* config, void* stream) {
  size_t need = 0;
  pkv_status st = pkv_attention_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                block_size, max_context_len, dtype, config, &need);
  if (st != PKV_OK) return st;
  PKV_CHECK(need <= PKV_NOALLOC_SCRATCH_BYTES, PKV_ERR_WORKSPACE_TOO_SMALL,
            "these sizes need %zu bytes of scratch; the fixed scratch holds %u bytes "
            "(use pkv_attention_decode with a larger workspace)",
            need, (unsigned)PKV_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != PKV_OK) return st;
  return pkv_attention_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                              max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                              block_size, num_blocks, scale, out, scratch,
                              PKV_NOALLOC_SCRATCH_BYTES, dtype, config, stream);
}

pkv_status pkv_attention_prefill_workspace_bytes(int32_t num_seqs, int32_t num_tokens,
                                                 int32_t max_query_len, int32_t max_context_len,
                                                 int32_t num_q_heads, int32_t num_kv_heads,
                                                 int32_t head_dim, int32_t block_size,
                                                 float scale, pkv_dtype dtype,
                                                 const pkv_attention_config* config,
                                                 size_t* bytes) {
  PKV_CHECK(bytes != nullptr, PKV_ERR_INVALID_ARGUMENT, "null bytes pointer");
  PrefillPlan plan;
  pkv_status st = plan_prefill(num_seqs, num_tokens, max_query_len, max_context_len, num_q_heads,
                               num_kv_heads, head_dim, block_size, 1, scale, dtype, config,
                               &plan);
  if (st != PKV_OK) return st;
  *bytes = plan.ws_bytes;
  return PKV_OK;
}

pkv_status pkv_attention_prefill(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* cu_seqlens, const int32_t* context_lens,
                                 int32_t num_seqs, int32_t num_tokens, int32_t max_query_len,
                                 int32_t max_context_len, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int64_t num_blocks, float scale, void* out, void* workspace,
                                 size_t workspace_bytes, pkv_dtype dtype,
                                 const pkv_attention_config* config, void* stream) {
  PKV_CHECK(max_blocks_per_seq >= 1, PKV_ERR_INVALID_ARGUMENT, "bad prefill sizes");
  PrefillPlan plan;
  pkv_status st = plan_prefill(num_seqs, num_tokens, max_query_len, max_context_len, num_q_heads,
                               num_kv_heads, head_dim, block_size, num_blocks, scale, dtype,
                               config, &plan);
  if (st != PKV_OK) return st;
  PKV_CHECK((int64_t)max_blocks_per_seq * block_size <= 2147483647, PKV_ERR_UNSUPPORTED,
            "table row too long");
  if (num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return PKV_OK;
  PKV_CHECK(q && k_cache && v_cache && block_tables && cu_seqlens && context_lens && out,
            PKV_ERR_INVALID_ARGUMENT, "null pointer");
  PKV_CHECK(aligned(k_cache, 16) && aligned(v_cache, 16) && aligned(q, 4) && aligned(out, 4),
            PKV_ERR_INVALID_ARGUMENT, "pools must be 16-byte aligned, q and out 4-byte aligned");
  PKV_CHECK(workspace_bytes >= plan.ws_bytes && (plan.ws_bytes == 0 || workspace != nullptr),
            PKV_ERR_WORKSPACE_TOO_SMALL, "prefill workspace: need %zu bytes", plan.ws_bytes);
  PKV_CHECK(plan.ws_bytes == 0 || aligned(workspace, 256), PKV_ERR_INVALID_ARGUMENT,
            "workspace must be 256-byte aligned");
  int dev = 0, sms = 0;
  st = device_facts(&dev, &sms);
  if (st != PKV_OK) return st;
  pkv::PfParams prm{};
  st = encode_pool_map(&prm.tmap_k, k_cache, num_blocks, block_size, num_kv_heads, head_dim);
  if (st != PKV_OK) return st;
  st = encode_pool_map(&prm.tmap_v, v_cache, num_blocks, block_size, num_kv_heads, head_dim);
  if (st != PKV_OK) return st;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.block_tables = block_tables;
  prm.cu_seqlens = cu_seqlens;
  prm.context_lens = context_lens;
  prm.num_blocks = num_blocks;
  prm.max_blocks_per_seq = max_blocks_per_seq;
  prm.num_seqs = num_seqs;
  prm.num_tokens = num_tokens;
  prm.max_len = max_context_len;
  prm.H_q = num_q_heads;
  prm.G = num_q_heads / num_kv_heads;
  prm.block_size = block_size;
  prm.scale_log2 = (float)((double)scale * 1.4426950408889634);
  if (plan.dec) {
    // several query rows per sequence through the stream-K decode kernel
    pkv::TcParams tp;
    memset(&tp, 0, sizeof(tp));
    tp.share_m = 1;
    st = encode_pool_map_heads(&tp.tmap_k, k_cache, num_blocks, block_size, num_kv_heads,
                               head_dim, plan.ap.hpc, false);
    if (st != PKV_OK) return st;
    st = encode_pool_map_heads(&tp.tmap_v, v_cache, num_blocks, block_size, num_kv_heads,
                               head_dim, plan.ap.hpc, false);
    if (st != PKV_OK) return st;
    tp.q = prm.q;
    tp.out = prm.out;
    tp.block_tables = block_tables;
    tp.context_lens = context_lens;
    tp.cu_seqlens = cu_seqlens;
    uint8_t* b = static_cast<uint8_t*>(workspace);
    const size_t T = (size_t)num_tokens;
    tp.ws.meta = reinterpret_cast<int4*>(b);
    b += align256(T * sizeof(int4));
    tp.ws.ml = reinterpret_cast<float2*>(b);
    b += align256(T * plan.ap.pmax * num_q_heads * sizeof(float2));
    tp.ws.o = reinterpret_cast<float*>(b);
    tp.ws.pmax = plan.ap.pmax;
    tp.num_blocks = num_blocks;
    tp.max_blocks_per_seq = max_blocks_per_seq;
    tp.num_seqs = num_seqs;
    tp.max_len = max_context_len;
    tp.H_q = num_q_heads;
    tp.G = num_q_heads / num_kv_heads;
    tp.block_size = block_size;
    tp.scale_log2 = prm.scale_log2;
    cudaStream_t strm = as_stream(stream);
    st = head_dim == 64
             ? launch_tc_d<64, 0>(plan.ap.hpc, block_size, tp, plan.ap.n_per_group,
                                  plan.ap.groups, strm, dev)
             : launch_tc_d<128, 0>(plan.ap.hpc, block_size, tp, plan.ap.n_per_group,
                                   plan.ap.groups, strm,
                                   dev);
    if (st != PKV_OK || plan.ap.pmax <= 1) return st;
    return launch_reduce<__nv_bfloat16>(head_dim, tp.ws, num_tokens, num_q_heads, out, strm);
  }
  prm.num_splits = plan.nsp;
  prm.split_tiles = plan.split_tiles;
  if (plan.nsp > 1) {
    uint8_t* b = static_cast<uint8_t*>(workspace);
    const size_t T = (size_t)num_tokens;
    prm.ws.meta = reinterpret_cast<int4*>(b);
    b += align256(T * sizeof(int4));
    prm.ws.ml = reinterpret_cast<float2*>(b);
    b += align256(T * plan.nsp * num_q_heads * sizeof(float2));
    prm.ws.o = reinterpret_cast<float*>(b);
    prm.ws.pmax = plan.nsp;
  }
  cudaStream_t strm = as_stream(stream);
  const int grid_x = (int)(plan.tiles * plan.nsp);
  if (plan.tc05) {
    // two query tiles per CTA sharing each K / V tile; one (SOLO) when every
    // (sequence, KV head) has a single tile
    const int pairs = (int)ceil_div(plan.tiles, 2);
    if (plan.tiles == 1) {
      if (head_dim == 128) return X2Inst<128, true>::launch(prm, 1, num_kv_heads, num_seqs, strm, dev);
      return X2Inst<64, true>::launch(prm, 1, num_kv_heads, num_seqs, strm, dev);
    }
    if (head_dim == 128) return X2Inst<128, false>::launch(prm, pairs, num_kv_heads, num_seqs, strm, dev);
    return X2Inst<64, false>::launch(prm, pairs, num_kv_heads, num_seqs, strm, dev);
  }
  const int nw = plan.nw;
  if (head_dim == 128) {
    st = nw == 1 ? PfInst<128, 1>::launch(prm, grid_x, num_kv_heads, num_seqs, strm, dev)
       : nw == 2 ? PfInst<128, 2>::launch(prm, grid_x, num_kv_heads, num_seqs, strm, dev)
                 : PfInst<128, 4>::launch(prm, grid_x, num_kv_heads, num_seqs, strm, dev);
  } else {
    st = nw == 1 ? PfInst<64, 1>::launch(prm, grid_x, num_kv_heads, num_seqs, strm, dev)
       : nw == 2 ? PfInst<64, 2>::launch(prm, grid_x, num_kv_heads, num_seqs, strm, dev)
                 : PfInst<64, 4>::launch(prm, grid_x, num_kv_heads, num_seqs, strm, dev);
  }
  if (st != PKV_OK || plan.nsp == 1) return st;
  // merge the key-range partials of every (token, head)
  return launch_reduce<__nv_bfloat16>(head_dim, prm.ws, num_tokens, num_q_heads, out, strm);
}

pkv_status pkv_kv_append_varlen(const void* k, const void* v, const int32_t* cu_seqlens,
                                const int32_t* context_lens, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, int32_t num_seqs, int32_t num_tokens,
                                void* k_cache, void* v_cache, int64_t num_blocks,
                                int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                pkv_dtype dtype, int64_t* slot_mapping_out, void* stream) {
  PKV_CHECK(num_seqs >= 0 && num_tokens >= 0 && max_blocks_per_seq >= 1 && num_blocks >= 1 &&
                block_size >= 1 && num_kv_heads >= 1 && head_dim >= 1 && dtype_ok(dtype),
            PKV_ERR_INVALID_ARGUMENT, "bad kv_append_varlen sizes");
  if (num_tokens == 0) return PKV_OK;
  PKV_CHECK(num_seqs >= 1, PKV_ERR_INVALID_ARGUMENT, "tokens without sequences");
  PKV_CHECK(k && v && cu_seqlens && context_lens && block_tables && k_cache && v_cache,
            PKV_ERR_INVALID_ARGUMENT, "null pointer");
  PKV_CHECK(num_blocks <= INT64_MAX / block_size, PKV_ERR_INVALID_ARGUMENT, "pool too large");
  const int64_t row = (int64_t)num_kv_heads * head_dim * elem_bytes(dtype);
  const int vw = vec_width(row, {k, v, k_cache, v_cache});
  PKV_CHECK(vw >= 2, PKV_ERR_INVALID_ARGUMENT, "misaligned rows");
  constexpr int threads = 128;
  const int64_t chunks = ceil_div(row / vw, threads);
  PKV_CHECK(chunks <= 65535, PKV_ERR_UNSUPPORTED, "rows too long");
  dim3 grid((unsigned)num_tokens, (unsigned)chunks, 2);
  cudaStream_t st = as_stream(stream);
  auto* kb = static_cast<const uint8_t*>(k);
  auto* vb = static_cast<const uint8_t*>(v);
  auto* kc = static_cast<uint8_t*>(k_cache);
  auto* vc = static_cast<uint8_t*>(v_cache);
#define PKV_APPEND_VARLEN(W)                                                                      \
  PKV_CUDA(launch_pdl(pkv::kv_append_varlen_kernel<W>, grid, dim3(threads), 0, st, kb, vb,       \
                      cu_seqlens, context_lens, num_seqs, block_tables, max_blocks_per_seq,     \
                      block_size, num_blocks, kc, vc, row, slot_mapping_out))
  switch (vw) {
    case 16: PKV_APPEND_VARLEN(16); break;
    case 8: PKV_APPEND_VARLEN(8); break;
    case 4: PKV_APPEND_VARLEN(4); break;
    default: PKV_APPEND_VARLEN(2); break;
  }
#undef PKV_APPEND_VARLEN
  return PKV_OK;
}

pkv_status pkv_get_device_error(int32_t* code, void* stream) {
  PKV_CHECK(code != nullptr, PKV_ERR_INVALID_ARGUMENT, "null code pointer");
  PKV_CUDA(cudaStreamSynchronize(as_stream(stream)));
  int h = 0;
  PKV_CUDA(cudaMemcpyFromSymbol(&h, pkv::g_error_word, sizeof(int)));
  *code = h;
  if (h != 0) {
    const int zero = 0;
    PKV_CUDA(cudaMemcpyToSymbol(pkv::g_error_word, &zero, sizeof(int)));
    return fail(PKV_ERR_DEVICE_CHECK, "device check failed with code %d", h);
  }
  return PKV_OK;
}

}  // extern "C"
