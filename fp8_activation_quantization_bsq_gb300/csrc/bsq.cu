// libbsq: host side of the C ABI declared in include/bsq.h -- argument
// validation, launch geometry, the TMA descriptor of the dense kernel, and the
// per-device error word.  All compute runs in the kernels of dense_quant.cuh,
// grouped_quant.cuh and interleave.cuh.
#include "bsq.h"

#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <algorithm>
#include <utility>

#include "block_scaled_dot.cuh"
#include "dense_quant.cuh"
#include "gemm_quant.cuh"
#include "device_common.cuh"
#include "grouped_quant.cuh"
#include "grouped_token.cuh"
#include "interleave.cuh"
#include "tensor_scale.cuh"

namespace {

using namespace bsq;

// Self-test of the bounded waits: an mbarrier that nothing arrives on is
// waited for with the same bounded wait the pipelined kernels use; it gives
// up after about a second and records BSQ_ERR_TIMEOUT.
__global__ void wait_timeout_selftest_kernel() {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0)) record_error(kErrTimeout);
}

constexpr int kDenseStages = 3;
constexpr int kMaxDevices = 64;
// Grouped quantize: groups averaging at most kGroupedLatencyMaxAvgRows rows
// (decode) take the row kernel (kRowsPerWarp destination rows per warp),
// larger groups (prefill) the band kernel (32 destination rows per block).
constexpr int64_t kGroupedLatencyMaxAvgRows = 16;
constexpr int kRowsPerWarp = 2;

struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int dense_ctas_per_sm[3] = {0, 0, 0};
  int tq_max_smem = 0;  // dynamic shared memory the token kernel may use
};

std::mutex g_mu;
DeviceInfo g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
bool g_encode_tried = false;

inline bool fmt_ok(int32_t f) { return f == BSQ_NVFP4 || f == BSQ_MXFP4 || f == BSQ_MXFP8; }
inline int sf_of(int32_t f) { return f == BSQ_NVFP4 ? 16 : 32; }
inline int atom_cols_of(int32_t f) { return 4 * sf_of(f); }
inline int64_t row_bytes_of(int32_t f, int64_t K) { return f == BSQ_MXFP8 ? K : K / 2; }
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Launch with programmatic stream serialization (programmatic dependent
// launch): the kernel may start while the previous kernel in the stream
// finishes; each kernel waits (griddepcontrol.wait) before touching memory.
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

template <int FMT>
void dense_kernel_setup(int fidx, DeviceInfo& d) {
  auto k = dense_quant_tma_kernel<FMT, kDenseStages>;
  const int smem = dense_smem_bytes<kDenseStages>();
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  int n = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kDenseThreads, smem);
  d.dense_ctas_per_sm[fidx] = n > 0 ? n : 1;
}

// Per-device constants, computed once with the device current.
bsq_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return BSQ_ERR_CUDA;
    dense_kernel_setup<kNVFP4>(0, d);
    dense_kernel_setup<kMXFP4>(1, d);
    dense_kernel_setup<kMXFP8>(2, d);
    cudaFuncSetAttribute(gemm_quant_kernel<kNVFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, gemm_smem_bytes());
    cudaFuncSetAttribute(gemm_quant_kernel<kMXFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, gemm_smem_bytes());
    cudaFuncSetAttribute(gemm_quant_kernel<kMXFP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, gemm_smem_bytes());
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    d.tq_max_smem = optin;
    cudaFuncSetAttribute(grouped_token_kernel<kNVFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, d.tq_max_smem);
    cudaFuncSetAttribute(grouped_token_kernel<kMXFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, d.tq_max_smem);
    cudaFuncSetAttribute(grouped_token_kernel<kMXFP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, d.tq_max_smem);
    if (cudaGetLastError() != cudaSuccess) return BSQ_ERR_CUDA;
    d.ready = true;
  }
  *out = &d;
  return BSQ_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode_tried) {
    g_encode_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode_tiled;
}

template <int FMT>
bsq_status launch_dense(const void* in, int64_t M, int64_t K, int64_t ld_in, void* out,
                        void* scales, float tsf, const float* tsf_dev, cudaStream_t stream) {
  DeviceInfo* d = nullptr;
  if (bsq_status s = device_info(&d); s != BSQ_OK) return s;
  auto enc = encode_tiled();
  if (!enc) return BSQ_ERR_CUDA;

  CUtensorMap map;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ld_in) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kDenseBoxCols),
                             static_cast<cuuint32_t>(kDenseTileRows)};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(in), gdim, gstride, box,
          estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return BSQ_ERR_CUDA;

  DenseArgs a;
  a.out = static_cast<uint8_t*>(out);
  a.scales = static_cast<uint8_t*>(scales);
  a.out_ld = row_bytes_of(FMT, K);
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.tiles_k = static_cast<int>(ceil_div(K, kDenseTileCols));
  a.num_tiles = static_cast<int>(ceil_div(M, kDenseTileRows) * a.tiles_k);
  a.kt_atoms = static_cast<int>(ceil_div(K, atom_cols_of(FMT)));
  a.vec32 = (a.out_ld % 32 == 0) && aligned(out, 32);
  a.tsf = tsf;
  a.tsf_dev = tsf_dev;

  const int fidx = FMT;
  const int64_t resident = static_cast<int64_t>(d->sm_count) * d->dense_ctas_per_sm[fidx];
  const int grid = static_cast<int>(a.num_tiles < resident ? a.num_tiles : resident);
  const cudaError_t e = launch_pdl(dense_quant_tma_kernel<FMT, kDenseStages>, dim3(grid),
                                   dim3(kDenseThreads), dense_smem_bytes<kDenseStages>(), stream,
                                   map, a);
  return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

template <int FMT, int KT>
bsq_status launch_grouped_rows(const GroupedArgs& a, cudaStream_t stream) {
  const int64_t chunks = ceil_div(a.kt_atoms, KT);
  const int64_t blocks = ceil_div(a.total_rows, static_cast<int64_t>(kGrWarps) * kRowsPerWarp);
  if (chunks > 65535 || blocks >= (int64_t(1) << 31)) return BSQ_ERR_SHAPE;
  if (blocks == 0) return BSQ_OK;
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(chunks));
  const cudaError_t e =
      launch_pdl(grouped_rows_kernel<FMT, KT, kRowsPerWarp>, grid, dim3(kGrThreads), 0, stream, a);
  return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

constexpr int kBdChunksPerBlock = 224;  // 32-element chunks per band-kernel block (a multiple of 32)

template <int FMT>
bsq_status launch_grouped_band(GroupedArgs a, cudaStream_t stream) {
  DeviceInfo* d = nullptr;
  if (bsq_status s = device_info(&d); s != BSQ_OK) return s;
  const int64_t c_pad = static_cast<int64_t>(a.kt_atoms) * (FMT == kNVFP4 ? 2 : 4);
  const int64_t blocks = ceil_div(a.total_rows, kBdRows);
  // a block runs along its 32 rows for up to kBdChunksPerBlock chunks; with
  // fewer rows the runs are split (multiples of 32 chunks) until the grid
  // holds about twelve blocks per SM.  Measured rotated without a gather,
  // K = 7168, NVFP4: 4096 rows 60.2 -> 18.2 us, 8192 rows 65.3 -> 32.7 us,
  // 16384 rows 64.0 -> 54.5 us, 32768 rows 103.6 -> 102.2 us (MXFP8 115.6 ->
  // 108.1 us); six blocks per SM instead gave 18.2 / 32.2 / 64.0 / 103.6 us.
  a.ktc = kBdChunksPerBlock;
  while (a.ktc > 32 && blocks * ceil_div(c_pad, static_cast<int64_t>(a.ktc)) < 12 * static_cast<int64_t>(d->sm_count) &&
         ceil_div(c_pad, static_cast<int64_t>(a.ktc - 32)) <= 65535)  // the grid's y extent
    a.ktc -= 32;
  const int64_t chunks = ceil_div(c_pad, a.ktc);
  if (chunks > 65535 || blocks >= (int64_t(1) << 31)) return BSQ_ERR_SHAPE;
  if (blocks == 0) return BSQ_OK;
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(chunks));
  const cudaError_t e = launch_pdl(grouped_band_kernel<FMT>, grid, dim3(32 * band_warps<FMT>()), 0, stream, a);
  return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

// One block per SM, the source rows split evenly; more blocks only when a
// block would own more than kTqMaxTokens rows.
template <int FMT>
bsq_status launch_grouped_token(const GroupedArgs& a, cudaStream_t stream) {
  DeviceInfo* d = nullptr;
  if (bsq_status s = device_info(&d); s != BSQ_OK) return s;
  // with no row_indices every destination row is its own source row, and
  // rows past in_rows still need their checks
  int64_t n_tok = a.row_indices != nullptr ? a.in_rows : std::max(a.in_rows, a.total_rows);
  n_tok = std::max<int64_t>(n_tok, 1);  // block 0 reports bad source rows
  int64_t blocks = std::min<int64_t>(d->sm_count, n_tok);
  if (ceil_div(n_tok, blocks) > kTqMaxTokens) blocks = ceil_div(n_tok, kTqMaxTokens);
  if (blocks >= (int64_t(1) << 31)) return BSQ_ERR_SHAPE;
  TqArgs q;
  q.n_tok = n_tok;
  q.tpb = static_cast<int>(ceil_div(n_tok, blocks));
  q.n_tab = (FMT == kNVFP4 && a.num_experts <= kTqTabExperts) ? a.num_experts : 0;
  // row_indices staging: two buffers of up to kTqStageInts entries in what
  // shared memory is left
  const size_t fixed = tq_smem_bytes(q.tpb, q.n_tab, 0);
  if (fixed + 8 * 16 > static_cast<size_t>(d->tq_max_smem)) return BSQ_ERR_SHAPE;
  const int64_t room = static_cast<int64_t>((static_cast<size_t>(d->tq_max_smem) - fixed) / 8) & ~int64_t(3);
  q.stage_ints = static_cast<int>(std::min<int64_t>(kTqStageInts, room));
  // few tokens per block: warps claim (token, step) units, the tokens'
  // descriptors kept in the staging area once the scan is done
  q.units = (q.tpb <= kTqUnitTokens &&
             static_cast<size_t>(q.stage_ints) * 8 >= static_cast<size_t>(q.tpb) * (kTqBucket * sizeof(TqDesc) + 4))
                ? 1 : 0;
  const size_t smem = tq_smem_bytes(q.tpb, q.n_tab, q.stage_ints);
  if (a.scale_ws != nullptr && ceil_div(a.kt_atoms, kIlvAtoms) > 65535) return BSQ_ERR_SHAPE;
  cudaError_t e = launch_pdl(grouped_token_kernel<FMT>, dim3(static_cast<unsigned>(blocks)), dim3(kTqThreads), smem,
                             stream, a, q);
  // scale rows staged in the workspace: to their 5D positions
  if (e == cudaSuccess && a.scale_ws != nullptr) {
    const dim3 grid(static_cast<unsigned>(a.total_scale_rows / 128),
                    static_cast<unsigned>(ceil_div(a.kt_atoms, kIlvAtoms)));
    // 16-byte staging loads when every staged row starts on a 16-byte boundary
    if (a.kt_atoms % 4 == 0)
      e = launch_pdl(grouped_scale_ws_kernel<16>, grid, dim3(kIlvThreads), 0, stream, a);
    else
      e = launch_pdl(grouped_scale_ws_kernel<4>, grid, dim3(kIlvThreads), 0, stream, a);
  }
  return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

// 2D TMA map of a K-major BF16 operand: rows x K, row stride ld elements,
// boxes of 64 elements (128 bytes, 128-byte swizzle) x box_rows rows; reads
// past the edges return zeros.
bool gemm_operand_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K, int64_t ld, uint32_t box_rows) {
  auto enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kGmBK), box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT>
bsq_status launch_gemm_quant(const GemmQuantArgs& p, const void* a, int64_t lda, const void* b, int64_t ldb,
                             cudaStream_t stream) {
  DeviceInfo* d = nullptr;
  if (bsq_status s = device_info(&d); s != BSQ_OK) return s;
  CUtensorMap ma, mb;
  if (!gemm_operand_map(&ma, a, p.M, p.K, lda, kGmBM) || !gemm_operand_map(&mb, b, p.N, p.K, ldb, kGmBN))
    return BSQ_ERR_CUDA;
  const int64_t tiles = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
  const int grid = static_cast<int>(std::min<int64_t>(tiles, d->sm_count));
  const cudaError_t e = launch_pdl(gemm_quant_kernel<FMT>, dim3(grid), dim3(kGmThreads), gemm_smem_bytes(), stream,
                                   ma, mb, p);
  return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

template <int FMT>
bsq_status launch_grouped(const GroupedArgs& a_in, int kt, int kernel, cudaStream_t stream) {
  GroupedArgs a = a_in;
  if (kernel == BSQ_GROUPED_AUTO) {
    if (a.total_rows <= kGroupedLatencyMaxAvgRows * a.G)
      kernel = BSQ_GROUPED_LATENCY;
    else if (a.row_indices != nullptr && a.G <= kTqMaxGroups && a.total_rows >= 2 * a.in_rows &&
             a.in_rows <= 8 * static_cast<int64_t>(a.K))
      // source rows reused: read each once.  Every block of the token
      // kernel scans all of row_indices (a few instructions per entry per
      // SM), which stays small next to the quantize for K >= 256 and
      // in_rows <= 8 K.
      kernel = BSQ_GROUPED_TOKEN;
    else
      kernel = BSQ_GROUPED_STREAM;
  }
  // the token kernel files destination rows as 32-bit indices
  if (kernel == BSQ_GROUPED_TOKEN && (a.G > kTqMaxGroups || a.total_rows >= (int64_t(1) << 32)))
    kernel = BSQ_GROUPED_STREAM;
  // the staging pays only for NVFP4 (per-destination scales: 8 atoms per
  // store of a step); MX and the other kernels store the scales in place
  if (FMT != kNVFP4) a.scale_ws = nullptr;
  if (kernel == BSQ_GROUPED_TOKEN) return launch_grouped_token<FMT>(a, stream);
  a.scale_ws = nullptr;
  if (kernel == BSQ_GROUPED_STREAM) return launch_grouped_band<FMT>(a, stream);
  if (kt == 0) {
    // automatic: the fewest atom columns per unit that still keep the grid
    // within four blocks per SM (fewer, larger units cost less to schedule
    // at decode sizes; more blocks than that gave nothing in the k sweeps)
    DeviceInfo* d = nullptr;
    if (bsq_status s = device_info(&d); s != BSQ_OK) return s;
    const int64_t row_blocks = ceil_div(a.total_rows, static_cast<int64_t>(kGrWarps) * kRowsPerWarp);
    kt = 8;
    for (int c : {1, 2, 4}) {
      if (row_blocks * ceil_div(a.kt_atoms, c) <= 4 * static_cast<int64_t>(d->sm_count)) {
        kt = c;
        break;
      }
    }
  }
  switch (kt) {
    case 1: return launch_grouped_rows<FMT, 1>(a, stream);
    case 2: return launch_grouped_rows<FMT, 2>(a, stream);
    case 4: return launch_grouped_rows<FMT, 4>(a, stream);
    default: return launch_grouped_rows<FMT, 8>(a, stream);
  }
}

}  // namespace

extern "C" {

int32_t bsq_version(void) { return (1 << 16) | 0; }

const char* bsq_status_string(int32_t s) {
  switch (s) {
    case BSQ_OK: return "BSQ_OK";
    case BSQ_ERR_NULL: return "BSQ_ERR_NULL: a required pointer is NULL";
    case BSQ_ERR_SHAPE: return "BSQ_ERR_SHAPE: invalid size or stride";
    case BSQ_ERR_ALIGN: return "BSQ_ERR_ALIGN: misaligned pointer or stride";
    case BSQ_ERR_VALUE: return "BSQ_ERR_VALUE: invalid scalar argument or device metadata";
    case BSQ_ERR_CUDA: return "BSQ_ERR_CUDA: a CUDA call failed";
    case BSQ_ERR_TIMEOUT: return "BSQ_ERR_TIMEOUT: a bounded device wait expired";
    default: return "unknown bsq status";
  }
}

int32_t bsq_block_size(int32_t fmt) { return fmt_ok(fmt) ? sf_of(fmt) : 0; }

int64_t bsq_packed_row_bytes(int32_t fmt, int64_t K) {
  if (!fmt_ok(fmt) || K < 0) return 0;
  return row_bytes_of(fmt, K);
}

int64_t bsq_scales5d_bytes(int32_t fmt, int64_t rows, int64_t K) {
  if (!fmt_ok(fmt) || rows < 0 || K < 0) return 0;
  return ceil_div(rows, 128) * ceil_div(K / sf_of(fmt), 4) * 512;
}

namespace {
bsq_status check_dense(int32_t fmt, const void* in, int64_t M, int64_t K, int64_t ld_in,
                       const void* out, const void* scales, bool* noop) {
  *noop = false;
  if (!fmt_ok(fmt)) return BSQ_ERR_VALUE;
  if (M < 0 || K < 0 || K % 32 != 0 || M >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
    return BSQ_ERR_SHAPE;
  if (M == 0 || K == 0) {
    *noop = true;
    return BSQ_OK;
  }
  if (ld_in < K) return BSQ_ERR_SHAPE;
  if (ceil_div(M, 128) * ceil_div(K, 128) >= (int64_t(1) << 31)) return BSQ_ERR_SHAPE;
  if (!in || !out || !scales) return BSQ_ERR_NULL;
  if (!aligned(in, 16) || !aligned(out, 16) || !aligned(scales, 16) || ld_in % 8 != 0)
    return BSQ_ERR_ALIGN;
  return BSQ_OK;
}

bsq_status dense_dispatch(int32_t fmt, const void* in, int64_t M, int64_t K, int64_t ld_in,
                          void* out, void* scales, float tsf, const float* tsf_dev,
                          cudaStream_t st) {
  switch (fmt) {
    case BSQ_NVFP4: return launch_dense<kNVFP4>(in, M, K, ld_in, out, scales, tsf, tsf_dev, st);
    case BSQ_MXFP4: return launch_dense<kMXFP4>(in, M, K, ld_in, out, scales, 1.0f, nullptr, st);
    default: return launch_dense<kMXFP8>(in, M, K, ld_in, out, scales, 1.0f, nullptr, st);
  }
}
}  // namespace

int32_t bsq_quantize(int32_t fmt, const void* in, int64_t M, int64_t K, int64_t ld_in, void* out,
                     void* scales, float tensor_sf, void* stream) {
  bool noop = false;
  if (bsq_status s = check_dense(fmt, in, M, K, ld_in, out, scales, &noop); s != BSQ_OK || noop)
    return s;
  if (fmt == BSQ_NVFP4 && !(std::isfinite(tensor_sf) && tensor_sf > 0.0f)) return BSQ_ERR_VALUE;
  return dense_dispatch(fmt, in, M, K, ld_in, out, scales, tensor_sf, nullptr,
                        static_cast<cudaStream_t>(stream));
}

int32_t bsq_quantize_dynamic(int32_t fmt, const void* in, int64_t M, int64_t K, int64_t ld_in,
                             void* out, void* scales, const float* tensor_sf_dev, void* stream) {
  bool noop = false;
  if (bsq_status s = check_dense(fmt, in, M, K, ld_in, out, scales, &noop); s != BSQ_OK || noop)
    return s;
  if (fmt == BSQ_NVFP4 && !tensor_sf_dev) return BSQ_ERR_NULL;
  if (fmt == BSQ_NVFP4 && !aligned(tensor_sf_dev, 4)) return BSQ_ERR_ALIGN;
  return dense_dispatch(fmt, in, M, K, ld_in, out, scales, 1.0f,
                        fmt == BSQ_NVFP4 ? tensor_sf_dev : nullptr,
                        static_cast<cudaStream_t>(stream));
}

int64_t bsq_tensor_sf_workspace_bytes(void) { return static_cast<int64_t>(sizeof(AmaxWorkspace)); }

int32_t bsq_tensor_sf(const void* in, int64_t M, int64_t K, int64_t ld_in, float* out,
                      void* workspace, int64_t workspace_bytes, void* stream) {
  if (M < 0 || K < 0 || K % 8 != 0 || K >= (int64_t(1) << 31)) return BSQ_ERR_SHAPE;
  if (M > 0 && K > 0 && ld_in < K) return BSQ_ERR_SHAPE;
  if (!out || !workspace || (M > 0 && K > 0 && !in)) return BSQ_ERR_NULL;
  if (workspace_bytes < static_cast<int64_t>(sizeof(AmaxWorkspace))) return BSQ_ERR_SHAPE;
  if (!aligned(out, 4) || !aligned(workspace, 16) || (M > 0 && K > 0 && (!aligned(in, 16) || ld_in % 8 != 0)))
    return BSQ_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  if (bsq_status s = device_info(&d); s != BSQ_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  AmaxWorkspace* ws = static_cast<AmaxWorkspace*>(workspace);
  const int64_t rows = (M > 0 && K > 0) ? M : 0;
  int64_t grid = ceil_div(rows, kAmaxWarps);
  // up to 8 blocks per SM (a warp per row on 8192 x 7168): with all rows in
  // flight at once the quantize that follows finds more of them in L2 (the
  // reads carry evict_last); the reduction alone is faster with 4 per SM
  // (20.3 against 22.5 us) but the tensor_sf -> quantize chain, its use, is
  // not (51.8 against 46.4 us)
  const int64_t cap = std::min<int64_t>(kAmaxMaxBlocks, static_cast<int64_t>(d->sm_count) * 8);
  grid = std::max<int64_t>(1, std::min(grid, cap));
  const cudaError_t e = launch_pdl(tensor_amax_kernel, dim3(static_cast<unsigned>(grid)),
                                   dim3(kAmaxThreads), 0, st, static_cast<const uint16_t*>(in), rows,
                                   static_cast<int>(K), ld_in, ws, out);
  return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

int64_t bsq_grouped_tensor_sf_workspace_bytes(int32_t num_experts) {
  if (num_experts < 1) return 0;
  return 16 + ceil_div(static_cast<int64_t>(num_experts) * 4, 16) * 16;
}

int32_t bsq_grouped_tensor_sf(const void* in, int64_t in_rows, int64_t K, int64_t ld_in,
                              const uint32_t* row_offsets, const int32_t* expert_ids,
                              const int32_t* row_indices, int32_t G, int64_t total_rows,
                              float* sf_out, int32_t num_experts, void* workspace,
                              int64_t workspace_bytes, void* stream) {
  if (num_experts < 1 || G < 0 || G > (1 << 20)) return BSQ_ERR_VALUE;
  if (in_rows < 0 || K < 0 || K % 8 != 0 || K >= (int64_t(1) << 31) || total_rows < 0)
    return BSQ_ERR_SHAPE;
  if (K > 0 && ld_in < K) return BSQ_ERR_SHAPE;
  if (workspace_bytes < bsq_grouped_tensor_sf_workspace_bytes(num_experts)) return BSQ_ERR_SHAPE;
  if (!sf_out || !workspace || (G > 0 && (!row_offsets || !expert_ids || (K > 0 && !in))))
    return BSQ_ERR_NULL;
  if (!aligned(sf_out, 4) || !aligned(workspace, 16) || !aligned(row_offsets, 4) ||
      !aligned(expert_ids, 4) || !aligned(row_indices, 4) ||
      (K > 0 && (!aligned(in, 16) || ld_in % 8 != 0)))
    return BSQ_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  if (bsq_status s = device_info(&d); s != BSQ_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int* counter = static_cast<unsigned int*>(workspace);
  unsigned int* amax_bits = counter + 4;
  GroupedAmaxArgs a;
  a.in = static_cast<const uint16_t*>(in);
  a.ld_in = ld_in;
  a.in_rows = in_rows;
  a.K = static_cast<int>(K);
  a.row_offsets = row_offsets;
  a.expert_ids = expert_ids;
  a.row_indices = row_indices;
  a.G = G;
  a.total_rows = (G > 0 && K > 0) ? total_rows : 0;
  a.num_experts = num_experts;
  a.amax_bits = amax_bits;
  a.counter = counter;
  a.sf = sf_out;
  // A gather that reuses source rows (row_indices, several destination rows
  // per source row): reduce each source row once, token-major, as long as
  // scanning row_indices once per 128 source rows stays under an eighth of
  // the gathered row bytes (in_rows <= 8 K) and the group metadata fits in
  // shared memory.
  const int64_t at_blocks = ceil_div(in_rows, kAtClusterTokens) * kAtCluster;
  if (row_indices != nullptr && G <= kAtMaxGroups && a.total_rows > in_rows && in_rows <= 8 * K &&
      in_rows > 0 && at_blocks < (int64_t(1) << 31)) {
    const int64_t blocks = at_blocks;
    const cudaError_t e = launch_pdl(grouped_amax_token_kernel, dim3(static_cast<unsigned>(blocks)),
                                     dim3(kAtThreads), 0, st, a);
    return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
  }
  int64_t grid = ceil_div(a.total_rows, kAmaxWarps);
  const int64_t cap = static_cast<int64_t>(d->sm_count) * 4;
  grid = std::max<int64_t>(1, std::min(grid, cap));
  const cudaError_t e = launch_pdl(grouped_amax_kernel, dim3(static_cast<unsigned>(grid)),
                                   dim3(kAmaxThreads), 0, st, a);
  return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

int32_t bsq_grouped_quantize_kernel(int32_t fmt, const void* in, int64_t in_rows, int64_t K,
                                    int64_t ld_in, const uint32_t* row_offsets,
                                    const uint32_t* scales_offsets, const int32_t* expert_ids,
                                    const float* sf, int32_t num_experts,
                                    const int32_t* row_indices, int32_t G, int64_t total_rows,
                                    int64_t total_scale_rows, void* out, void* scales,
                                    int32_t k_tiles_per_block, int32_t kernel, void* stream) {
  return bsq_grouped_quantize_ws(fmt, in, in_rows, K, ld_in, row_offsets, scales_offsets, expert_ids, sf,
                                 num_experts, row_indices, G, total_rows, total_scale_rows, out, scales,
                                 k_tiles_per_block, kernel, nullptr, 0, stream);
}

int64_t bsq_grouped_quantize_workspace_bytes(int32_t fmt, int64_t total_scale_rows, int64_t K) {
  if (!fmt_ok(fmt) || total_scale_rows < 0 || K < 0) return 0;
  // staged scale rows, then one int32 per 128-row band
  return total_scale_rows * ceil_div(K / sf_of(fmt), 4) * 4 + ceil_div(total_scale_rows / 128 * 4, 16) * 16;
}

int32_t bsq_grouped_quantize_ws(int32_t fmt, const void* in, int64_t in_rows, int64_t K, int64_t ld_in,
                                const uint32_t* row_offsets, const uint32_t* scales_offsets,
                                const int32_t* expert_ids, const float* sf, int32_t num_experts,
                                const int32_t* row_indices, int32_t G, int64_t total_rows,
                                int64_t total_scale_rows, void* out, void* scales, int32_t k_tiles_per_block,
                                int32_t kernel, void* workspace, int64_t workspace_bytes, void* stream) {
  if (!fmt_ok(fmt)) return BSQ_ERR_VALUE;
  if (k_tiles_per_block != 0 && k_tiles_per_block != 1 && k_tiles_per_block != 2 && k_tiles_per_block != 4 &&
      k_tiles_per_block != 8)
    return BSQ_ERR_VALUE;
  if (kernel != BSQ_GROUPED_AUTO && kernel != BSQ_GROUPED_STREAM && kernel != BSQ_GROUPED_LATENCY &&
      kernel != BSQ_GROUPED_TOKEN)
    return BSQ_ERR_VALUE;
  if (G < 0 || G > (1 << 20)) return BSQ_ERR_VALUE;
  if (in_rows < 0 || K < 0 || K % 32 != 0 || K >= (int64_t(1) << 31) || total_rows < 0 ||
      total_scale_rows < 0 || total_scale_rows % 128 != 0 ||
      total_scale_rows / 128 >= (int64_t(1) << 31))
    return BSQ_ERR_SHAPE;
  if (G == 0 || K == 0 || total_scale_rows == 0) return BSQ_OK;
  if (ld_in < K) return BSQ_ERR_SHAPE;
  if (!in || !row_offsets || !scales_offsets || !expert_ids || !out || !scales) return BSQ_ERR_NULL;
  if (fmt == BSQ_NVFP4 && !sf) return BSQ_ERR_NULL;
  if (fmt == BSQ_NVFP4 && num_experts < 1) return BSQ_ERR_VALUE;
  if (!aligned(in, 16) || ld_in % 8 != 0 || !aligned(out, 16) || !aligned(scales, 16) ||
      !aligned(row_offsets, 4) || !aligned(scales_offsets, 4) || !aligned(expert_ids, 4) ||
      !aligned(sf, 4) || !aligned(row_indices, 4) || !aligned(workspace, 16))
    return BSQ_ERR_ALIGN;
  if (workspace != nullptr && workspace_bytes < bsq_grouped_quantize_workspace_bytes(fmt, total_scale_rows, K))
    return BSQ_ERR_SHAPE;

  GroupedArgs a{};
  a.scale_ws = static_cast<uint8_t*>(workspace);
  a.in = static_cast<const uint16_t*>(in);
  a.ld_in = ld_in;
  a.in_rows = in_rows;
  a.K = static_cast<int>(K);
  a.row_offsets = row_offsets;
  a.scales_offsets = scales_offsets;
  a.expert_ids = expert_ids;
  a.sf = fmt == BSQ_NVFP4 ? sf : nullptr;
  a.num_experts = num_experts;
  a.row_indices = row_indices;
  a.G = G;
  a.total_rows = total_rows;
  a.total_scale_rows = total_scale_rows;
  a.out = static_cast<uint8_t*>(out);
  a.out_ld = row_bytes_of(fmt, K);
  a.scales = static_cast<uint8_t*>(scales);
  a.kt_atoms = static_cast<int>(ceil_div(K, atom_cols_of(fmt)));
  a.in_vec32 = aligned(in, 32) && ld_in % 16 == 0;
  a.out_vec32 = aligned(out, 32) && a.out_ld % 32 == 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (fmt) {
    case BSQ_NVFP4: return launch_grouped<kNVFP4>(a, k_tiles_per_block, kernel, st);
    case BSQ_MXFP4: return launch_grouped<kMXFP4>(a, k_tiles_per_block, kernel, st);
    default: return launch_grouped<kMXFP8>(a, k_tiles_per_block, kernel, st);
  }
}

int32_t bsq_grouped_quantize(int32_t fmt, const void* in, int64_t in_rows, int64_t K,
                             int64_t ld_in, const uint32_t* row_offsets,
                             const uint32_t* scales_offsets, const int32_t* expert_ids,
                             const float* sf, int32_t num_experts, const int32_t* row_indices,
                             int32_t G, int64_t total_rows, int64_t total_scale_rows, void* out,
                             void* scales, int32_t k_tiles_per_block, void* stream) {
  return bsq_grouped_quantize_kernel(fmt, in, in_rows, K, ld_in, row_offsets, scales_offsets,
                                     expert_ids, sf, num_experts, row_indices, G, total_rows,
                                     total_scale_rows, out, scales, k_tiles_per_block,
                                     BSQ_GROUPED_AUTO, stream);
}

int32_t bsq_gemm_quantize(int32_t fmt, const void* a, const void* b, int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldb, float tensor_sf, void* out, void* scales5d, void* c_bf16,
                          void* stream) {
  if (!fmt_ok(fmt)) return BSQ_ERR_VALUE;
  if (M < 0 || N < 0 || K < 0 || N % 128 != 0 || K % 32 != 0 || N >= (int64_t(1) << 31) ||
      K >= (int64_t(1) << 31))
    return BSQ_ERR_SHAPE;
  if (M == 0 || N == 0) return BSQ_OK;
  if (K == 0 || lda < K || ldb < K) return BSQ_ERR_SHAPE;
  if (!a || !b || !out || !scales5d) return BSQ_ERR_NULL;
  if (!aligned(a, 16) || !aligned(b, 16) || lda % 8 != 0 || ldb % 8 != 0 || !aligned(out, 16) ||
      !aligned(scales5d, 16) || !aligned(c_bf16, 16))
    return BSQ_ERR_ALIGN;
  if (fmt == BSQ_NVFP4 && !(std::isfinite(tensor_sf) && tensor_sf > 0.0f)) return BSQ_ERR_VALUE;
  if (ceil_div(M, kGmBM) * ceil_div(N, kGmBN) >= (int64_t(1) << 31) || M >= (int64_t(1) << 31)) return BSQ_ERR_SHAPE;
  GemmQuantArgs p{};
  p.M = M;
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.tiles_m = static_cast<int>(ceil_div(M, kGmBM));
  p.tiles_n = static_cast<int>(ceil_div(N, kGmBN));
  p.tsf = fmt == BSQ_NVFP4 ? tensor_sf : 1.0f;
  p.out = static_cast<uint8_t*>(out);
  p.out_ld = row_bytes_of(fmt, N);
  p.scales = static_cast<uint8_t*>(scales5d);
  p.kt_atoms = static_cast<int>(N / atom_cols_of(fmt));
  p.c = static_cast<uint16_t*>(c_bf16);
  p.vec32 = aligned(out, 32) && p.out_ld % 32 == 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (fmt) {
    case BSQ_NVFP4: return launch_gemm_quant<kNVFP4>(p, a, lda, b, ldb, st);
    case BSQ_MXFP4: return launch_gemm_quant<kMXFP4>(p, a, lda, b, ldb, st);
    default: return launch_gemm_quant<kMXFP8>(p, a, lda, b, ldb, st);
  }
}

int32_t bsq_scales_interleave(const void* scales2d, int64_t M, int64_t S, int64_t ld,
                              void* scales5d, void* stream) {
  if (M < 0 || S < 0) return BSQ_ERR_SHAPE;
  if (M == 0 || S == 0) return BSQ_OK;
  if (ld < S) return BSQ_ERR_SHAPE;
  const int64_t bands = ceil_div(M, 128), kt_atoms = ceil_div(S, 4);
  const int64_t chunks = ceil_div(kt_atoms, kIlvAtoms);
  if (bands >= (int64_t(1) << 31) || chunks > 65535 || kt_atoms >= (int64_t(1) << 31))
    return BSQ_ERR_SHAPE;
  if (!scales2d || !scales5d) return BSQ_ERR_NULL;
  if (!aligned(scales5d, 16)) return BSQ_ERR_ALIGN;
  const uint8_t* in = static_cast<const uint8_t*>(scales2d);
  uint8_t* out = static_cast<uint8_t*>(scales5d);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  dim3 grid(static_cast<unsigned>(bands), static_cast<unsigned>(chunks));
  const int ikt = static_cast<int>(kt_atoms);
  cudaError_t e;
  if (aligned(in, 16) && ld % 16 == 0 && S % 16 == 0)
    e = launch_pdl(interleave_kernel<16>, grid, dim3(kIlvThreads), 0, st, in, M, S, ld, out, ikt);
  else if (aligned(in, 4) && ld % 4 == 0 && S % 4 == 0)
    e = launch_pdl(interleave_kernel<4>, grid, dim3(kIlvThreads), 0, st, in, M, S, ld, out, ikt);
  else
    e = launch_pdl(interleave_kernel<1>, grid, dim3(kIlvThreads), 0, st, in, M, S, ld, out, ikt);
  return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

int32_t bsq_block_scaled_dot(int32_t fmt, const void* a_packed, const void* a_scales5d, float a_tsf,
                             const void* b_packed, const void* b_scales5d, float b_tsf, int64_t M,
                             int64_t N, int64_t K, double* c_out, void* stream) {
  if (!fmt_ok(fmt)) return BSQ_ERR_VALUE;
  if (M < 0 || N < 0 || K < 0 || K % 32 != 0 || K >= (int64_t(1) << 31) || M >= (int64_t(1) << 35) ||
      N >= (int64_t(1) << 35))
    return BSQ_ERR_SHAPE;
  if (M == 0 || N == 0) return BSQ_OK;
  if (!c_out || (K > 0 && (!a_packed || !a_scales5d || !b_packed || !b_scales5d))) return BSQ_ERR_NULL;
  if (!aligned(c_out, 8)) return BSQ_ERR_ALIGN;
  if (fmt == BSQ_NVFP4 && !(std::isfinite(a_tsf) && a_tsf > 0.0f && std::isfinite(b_tsf) && b_tsf > 0.0f))
    return BSQ_ERR_VALUE;
  const double inv_tsf = fmt == BSQ_NVFP4 ? 1.0 / (static_cast<double>(a_tsf) * b_tsf) : 1.0;
  const int64_t gx = ceil_div(N, 16), gy = ceil_div(M, 16);
  if (gx >= (int64_t(1) << 31) || gy > 65535) return BSQ_ERR_SHAPE;
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const auto* ap = static_cast<const uint8_t*>(a_packed);
  const auto* sap = static_cast<const uint8_t*>(a_scales5d);
  const auto* bp = static_cast<const uint8_t*>(b_packed);
  const auto* sbp = static_cast<const uint8_t*>(b_scales5d);
  const int k = static_cast<int>(K);
  cudaError_t e;
  switch (fmt) {
    case BSQ_NVFP4:
      e = launch_pdl(block_scaled_dot_kernel<kNVFP4>, grid, dim3(256), 0, st, ap, sap, bp, sbp, M, N, k, inv_tsf, c_out);
      break;
    case BSQ_MXFP4:
      e = launch_pdl(block_scaled_dot_kernel<kMXFP4>, grid, dim3(256), 0, st, ap, sap, bp, sbp, M, N, k, inv_tsf, c_out);
      break;
    default:
      e = launch_pdl(block_scaled_dot_kernel<kMXFP8>, grid, dim3(256), 0, st, ap, sap, bp, sbp, M, N, k, inv_tsf, c_out);
  }
  return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

int32_t bsq_selftest_wait_timeout(void* stream) {
  const cudaError_t e = launch_pdl(wait_timeout_selftest_kernel, dim3(1), dim3(32), 0,
                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

int32_t bsq_device_error(void* stream, int32_t* code_out) {
  if (!code_out) return BSQ_ERR_NULL;
  *code_out = BSQ_OK;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return BSQ_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v)) != cudaSuccess) return BSQ_ERR_CUDA;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return BSQ_ERR_CUDA;
  }
  *code_out = static_cast<int32_t>(v);
  return BSQ_OK;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Per-expert tensor scales without caller-provided scratch.
//
// Some callers have no way to obtain device memory at the point where they
// need the scales: a plugin whose C interface passes only input and output
// pointers, a host framework that owns every device allocation through its
// own pool and forbids raw cudaMalloc, or a latency-critical loop that cannot
// afford the device-wide synchronization cudaMalloc/cudaFree may imply.  For
// them the reduction's scratch (a completion counter and one running maximum
// per expert) lives in the file-scope array below, one copy per device that
// loads this library, held until the process exits.  Host code must not use
// the array's name as a device address: it is a host-side stand-in, and only
// the address cudaGetSymbolAddress returns for the current device is valid.
namespace {

constexpr int kNoAllocScratchWords = 4 + BSQ_NOALLOC_MAX_EXPERTS;  // counter (+3 pad) | maxima
static __device__ __align__(256) unsigned int g_noalloc_scratch[kNoAllocScratchWords];

struct NoAllocDevice {
  bool ready = false;
  unsigned int* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int sm_count = 0;
};

std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_devices[kMaxDevices];

// Once per device, with that device current: look up the array's device
// address and the SM count.
bsq_status noalloc_device(NoAllocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_devices[dev];
  if (!d.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return BSQ_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return BSQ_ERR_CUDA;
    d.scratch = static_cast<unsigned int*>(ptr);
    d.ready = true;
  }
  *out = &d;
  return BSQ_OK;
}

}  // namespace

extern "C" {

int32_t bsq_grouped_tensor_sf_noalloc(const void* in, int64_t in_rows, int64_t K, int64_t ld_in,
                                      const uint32_t* row_offsets, const int32_t* expert_ids,
                                      const int32_t* row_indices, int32_t G, int64_t total_rows,
                                      float* sf_out, int32_t num_experts, void* stream) {
  if (num_experts < 1 || G < 0 || G > (1 << 20)) return BSQ_ERR_VALUE;
  if (num_experts > BSQ_NOALLOC_MAX_EXPERTS) return BSQ_ERR_SHAPE;  // beyond the static scratch
  if (in_rows < 0 || K < 0 || K % 8 != 0 || K >= (int64_t(1) << 31) || total_rows < 0)
    return BSQ_ERR_SHAPE;
  if (K > 0 && ld_in < K) return BSQ_ERR_SHAPE;
  if (!sf_out || (G > 0 && (!row_offsets || !expert_ids || (K > 0 && !in)))) return BSQ_ERR_NULL;
  if (!aligned(sf_out, 4) || !aligned(row_offsets, 4) || !aligned(expert_ids, 4) ||
      !aligned(row_indices, 4) || (K > 0 && (!aligned(in, 16) || ld_in % 8 != 0)))
    return BSQ_ERR_ALIGN;
  NoAllocDevice* d = nullptr;
  if (bsq_status s = noalloc_device(&d); s != BSQ_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's counter and maxima: zero the part
  // this call uses (counter, padding and num_experts maxima).
  const size_t clear_bytes = static_cast<size_t>(16 + 4 * static_cast<int64_t>(num_experts));
  if (cudaMemsetAsync(d->scratch, 0, clear_bytes, st) != cudaSuccess) return BSQ_ERR_CUDA;
  GroupedAmaxArgs a;
  a.in = static_cast<const uint16_t*>(in);
  a.ld_in = ld_in;
  a.in_rows = in_rows;
  a.K = static_cast<int>(K);
  a.row_offsets = row_offsets;
  a.expert_ids = expert_ids;
  a.row_indices = row_indices;
  a.G = G;
  a.total_rows = (G > 0 && K > 0) ? total_rows : 0;
  a.num_experts = num_experts;
  a.amax_bits = d->scratch + 4;
  a.counter = d->scratch;
  a.sf = sf_out;
  int64_t grid = ceil_div(a.total_rows, kAmaxWarps);
  grid = std::max<int64_t>(1, std::min<int64_t>(grid, static_cast<int64_t>(d->sm_count) * 4));
  const cudaError_t e = launch_pdl(grouped_amax_kernel, dim3(static_cast<unsigned>(grid)),
                                   dim3(kAmaxThreads), 0, st, a);
  return e == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

}  // extern "C"
