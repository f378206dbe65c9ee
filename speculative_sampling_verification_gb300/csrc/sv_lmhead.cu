// The scoring step's final projection fused with the row statistics of the
// temperature transform ("Accelerating Large Language Model Decoding with
// Speculative Sampling", wikillm.com paper card: Algorithm 2 step 2, one
// target call scores the K+1 prefixes; §4.1 "Why it works (conditional
// scoring)"; §4.2 "Decoding transforms").
//
// For hidden states h [N, D] and the projection's weight W [V, D] (one row per
// token, bf16), the logits l = h W^T are formed on the tensor cores and never
// leave the chip. The output is cut into 128 x 256 tiles of l (128 rows of h,
// 256 tokens); one persistent CTA per SM takes tiles blockIdx.x,
// blockIdx.x + gridDim.x, ... (the 128-row tiles that share 256 tokens are
// consecutive, so a slice of W is read from HBM about once). A tile is
// accumulated in tensor memory over D with tcgen05.mma (bf16 operands staged
// in shared memory by TMA, fp32 accumulator in TMEM); its epilogue reduces it
// to one (max, sum) pair per row, sum of 2^((l - max) log2(e)/T), and picks up
// the logit at the row's token when that token falls in the tile. A second
// kernel combines the pairs of a row into max_i l_i/T and log sum_i exp(l_i/T).
//
// Warp roles in a CTA of 192 threads: warps 0-3 read the accumulator (warp w
// owns TMEM lanes 32w .. 32w+31, i.e. rows 32w .. 32w+31 of the tile); warp 4
// issues the TMA loads; warp 5 allocates the tensor memory and issues the
// MMAs. Four shared-memory stages of 48 KB (a 128 x 64 tile of h and a
// 256 x 64 tile of W), refilled across tile boundaries, with full/empty
// mbarriers; two accumulators of 256 TMEM columns, so that the epilogue of one
// tile runs while the MMAs of the next fill the other (full/empty mbarriers
// between the MMA warp and the epilogue warps). Every wait is bounded: one
// that runs out sets a status bit and ends the CTA's work, after which the
// tensor memory is still released.
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/spec_verify.h"
#include "sv_device.cuh"

namespace sv {
namespace lmh {

constexpr int kBM = 128;             // rows of h per tile (MMA M)
constexpr int kBN = 256;             // tokens per tile (MMA N)
constexpr int kBK = 64;              // D per stage: 128 bytes of bf16, one swizzle atom
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kTileA = kBM * kBK * 2;   // 16 KB
constexpr int kTileB = kBN * kBK * 2;   // 32 KB
constexpr int kStageBytes = kTileA + kTileB;
constexpr int kAccs = 2;                // accumulators (TMEM buffers)
constexpr int kTmemCols = 256 * kAccs;  // each 128 x 256 fp32
constexpr unsigned kDevTimeout = 256;

// Dynamic shared memory: the stages (1024-byte aligned for the 128-byte
// swizzle), then the barriers and the tensor-memory address.
struct Tail {
  unsigned long long full[kStages];
  unsigned long long empty[kStages];
  unsigned long long acc_full[kAccs];   // an accumulator's MMAs are complete
  unsigned long long acc_empty[kAccs];  // the epilogue has read an accumulator
  unsigned tmem_base;
  unsigned abort;
};
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /* alignment slack */ + (int)sizeof(Tail);

struct Args {
  const int32_t* tokens;
  int N, D, V, n_mt, n_nt, nk, n_tiles;
  float c2;          // log2(e)/T
  float2* part;      // [N, n_nt] (max l, sum 2^((l - max) c2)) per row and tile
  float* at;         // [N] l at the row's token
  unsigned* status;
};

// ---------------------------------------------------------------- PTX wrappers

SV_DEVINL unsigned smem_addr(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

SV_DEVINL void mbar_init(unsigned bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

SV_DEVINL void mbar_expect_tx(unsigned bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

SV_DEVINL void mbar_arrive(unsigned bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

SV_DEVINL bool mbar_try_wait(unsigned bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with `parity` to complete. Gives up (returning
// false, after setting the status bit and the CTA's abort flag) after the
// common wall-time limit, or at once when another thread of the CTA gave up.
SV_DEVINL bool mbar_wait(unsigned bar, unsigned parity, volatile unsigned* abort,
                         unsigned* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (unsigned i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 0) {
      if (*abort) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        atomicOr(status, kDevTimeout);
        *abort = 1;
        return false;
      }
    }
  }
}

SV_DEVINL void tma_load_2d(unsigned dst, const CUtensorMap* map, int x, int y, unsigned bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Shared-memory descriptor of a K-major bf16 tile whose rows are 128 bytes
// with the 128-byte swizzle (what TMA writes with CU_TENSOR_MAP_SWIZZLE_128B):
// start address >> 4 in bits 0-13, leading byte offset 16 B (>> 4 = 1) in
// bits 16-29 (not used by this layout), stride byte offset 1024 B (8 rows of
// 128 B) >> 4 in bits 32-45, descriptor version 1 in bits 46-47, base offset
// 0 (tiles are 1024-byte aligned), swizzle mode 2 (128 B) in bits 61-63.
SV_DEVINL uint64_t smem_desc_sw128(unsigned addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
// (bits 7-9 = 1) and B (bits 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

SV_DEVINL void mma_bf16(unsigned tmem_d, uint64_t a, uint64_t b, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(kIdesc), "r"((unsigned)accumulate)
      : "memory");
}

SV_DEVINL void mma_commit(unsigned bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

SV_DEVINL void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SV_DEVINL void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
SV_DEVINL void tmem_ld32(unsigned taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- the GEMM + statistics kernel

__global__ void __launch_bounds__(kThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_w,
                  Args a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Tail* tail = reinterpret_cast<Tail*>(smem + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&tail->full[s]), 1);
      mbar_init(smem_addr(&tail->empty[s]), 1);
    }
    for (int i = 0; i < kAccs; ++i) {
      mbar_init(smem_addr(&tail->acc_full[i]), 1);   // one tcgen05.commit
      mbar_init(smem_addr(&tail->acc_empty[i]), 4);  // one arrival per epilogue warp
    }
    tail->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 4 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_h)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_w)) : "memory");
  }
  if (warp == 5) {  // the whole warp allocates the accumulators' columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tail->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const unsigned tmem = tail->tmem_base;
  volatile unsigned* abort = &tail->abort;
  const int first = blockIdx.x, step = gridDim.x;

  if (warp == 4) {
    // TMA producer: the k-blocks of this CTA's tiles, one ring across tiles.
    if (lane == 0) {
      unsigned it = 0;
      bool ok = true;
      for (int t = first; t < a.n_tiles && ok; t += step) {
        const int m0 = (t % a.n_mt) * kBM, n0 = (t / a.n_mt) * kBN;
        for (int kb = 0; kb < a.nk; ++kb, ++it) {
          const int s = (int)(it % kStages);
          const unsigned ph = (it / kStages) & 1u;
          if (it >= kStages && !mbar_wait(smem_addr(&tail->empty[s]), ph ^ 1u, abort, a.status)) {
            ok = false;
            break;
          }
          const unsigned full = smem_addr(&tail->full[s]);
          mbar_expect_tx(full, kStageBytes);
          const unsigned dst = smem_addr(smem + s * kStageBytes);
          tma_load_2d(dst, &map_h, kb * kBK, m0, full);
          tma_load_2d(dst + kTileA, &map_w, kb * kBK, n0, full);
        }
      }
    }
  } else if (warp == 5) {
    // MMA issuer: per tile, an accumulator the epilogue has released, four
    // K = 16 steps per stage; a stage goes back to the producer when its MMAs
    // complete, and the accumulator to the epilogue when the tile's last does.
    if (lane == 0) {
      unsigned it = 0, ti = 0;
      bool ok = true;
      for (int t = first; t < a.n_tiles && ok; t += step, ++ti) {
        const unsigned acc = ti % kAccs, aph = (ti / kAccs) & 1u;
        if (ti >= kAccs && !mbar_wait(smem_addr(&tail->acc_empty[acc]), aph ^ 1u, abort, a.status))
          break;
        tmem_fence_after();
        const unsigned d = tmem + acc * 256;
        for (int kb = 0; kb < a.nk; ++kb, ++it) {
          const int s = (int)(it % kStages);
          const unsigned ph = (it / kStages) & 1u;
          if (!mbar_wait(smem_addr(&tail->full[s]), ph, abort, a.status)) {
            ok = false;
            break;
          }
          tmem_fence_after();
          const unsigned sa = smem_addr(smem + s * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t da = smem_desc_sw128(sa + kk * 32);
            const uint64_t db = smem_desc_sw128(sa + kTileA + kk * 32);
            mma_bf16(d, da, db, kb > 0 || kk > 0);
          }
          mma_commit(smem_addr(&tail->empty[s]));
        }
        if (ok) mma_commit(smem_addr(&tail->acc_full[acc]));
      }
    }
  } else {
    // Epilogue: thread (warp, lane) owns row 32 warp + lane of each tile.
    unsigned ti = 0;
    for (int t = first; t < a.n_tiles; t += step, ++ti) {
      const unsigned acc = ti % kAccs, aph = (ti / kAccs) & 1u;
      const int mt = t % a.n_mt, nt = t / a.n_mt;
      const int m0 = mt * kBM, n0 = nt * kBN;
      const int row = m0 + warp * 32 + lane;
      // tcgen05.ld is warp-wide: the warp reads the accumulator only if every
      // lane saw it complete.
      const bool ok =
          __all_sync(0xffffffffu, mbar_wait(smem_addr(&tail->acc_full[acc]), aph, abort, a.status));
      if (!ok) break;
      tmem_fence_after();
      const int tok = row < a.N ? __ldg(a.tokens + row) : -1;
      const int tcol = tok - n0;  // the token's column in this tile, if in [0, 256)
      float mx = -INFINITY, hmx = -INFINITY, sum = 0.0f, at = 0.0f;
      bool have_at = false;
      const unsigned tbase = tmem + acc * 256 + ((unsigned)(warp * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        float v[32];
        tmem_ld32(tbase + (unsigned)(c * 32), v);
        const int col0 = n0 + c * 32;
        float cm = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (col0 + j >= a.V) v[j] = -INFINITY;  // padding columns of the last tile
          cm = fmaxf(cm, v[j]);
        }
        if (tcol >= c * 32 && tcol < c * 32 + 32) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (tcol - c * 32 == j) at = v[j];
          have_at = true;
        }
        if (cm > mx) {
          const float h = cm * a.c2;
          if (mx != -INFINITY) sum *= ex2_fast(hmx - h);
          mx = cm;
          hmx = h;
        }
        if (mx != -INFINITY) {
#pragma unroll
          for (int j = 0; j < 32; ++j) sum += ex2_fast(__fmaf_rn(v[j], a.c2, -hmx));
        }
      }
      // The accumulator is read: hand it back to the MMA warp.
      tmem_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&tail->acc_empty[acc]));
      // 2^(hmx - mx c2) folds the rounding of hmx back in (to first order).
      if (mx != -INFINITY) sum *= __fmaf_rn(__fmaf_rn(-mx, a.c2, hmx), 0.69314718f, 1.0f);
      if (row < a.N) {
        a.part[(size_t)row * a.n_nt + nt] = make_float2(mx, sum);
        if (have_at && tok < a.V) a.at[row] = at;
      }
    }
  }
  tmem_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();  // dealloc is warp-wide: re-converge after lane 0's MMA loop
    tmem_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// One warp per row: the row's tile pairs combined into max l/T and the
// log-sum-exp, in fp64; rows without a token in [0, V) get at = NaN.
__global__ void lmhead_combine_kernel(Args a, double inv_t_d, double* row_max, double* lse) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.N) return;
  const float2* p = a.part + (size_t)row * a.n_nt;
  float m = -INFINITY;
  for (int t = lane; t < a.n_nt; t += 32) m = fmaxf(m, p[t].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  double s = 0.0;
  for (int t = lane; t < a.n_nt; t += 32) {
    const float2 q = p[t];
    if (q.x != -INFINITY) s += (double)q.y * exp2(((double)q.x - (double)m) * (double)a.c2);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) {
    const bool bad = !(m > -INFINITY) || !(s > 0.0) || !(s < INFINITY);
    if (bad) atomicOr(a.status, 32u);  // a non-finite logit
    row_max[row] = bad ? __longlong_as_double(0x7ff8000000000000LL) : (double)m * inv_t_d;
    lse[row] = bad ? __longlong_as_double(0x7ff8000000000000LL) : (double)m * inv_t_d + log(s);
    const int tok = a.tokens[row];
    if (tok < 0 || tok >= a.V) a.at[row] = __int_as_float(0x7fc00000);
  }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A [rows, D] bf16 row-major matrix as TMA boxes of kBK x box_rows, with the
// 128-byte swizzle; reads outside the matrix (rows >= rows, columns >= D)
// fill with zeros.
bool make_map(CUtensorMap* m, const void* base, int rows, int D, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace lmh
}  // namespace sv

using namespace sv::lmh;

namespace {

bool lmhead_sizes(int N, int D, int V, int* n_mt, int* n_nt, size_t* bytes) {
  if (N < 0 || D < 8 || D % 8 != 0 || V < 1 || D > (1 << 20) || V > (1 << 30)) return false;
  if ((long long)N * D > (1ll << 40)) return false;
  *n_mt = (N + kBM - 1) / kBM;
  *n_nt = (V + kBN - 1) / kBN;
  *bytes = 256 + (size_t)N * (size_t)(*n_nt) * sizeof(float2);
  return true;
}

bool misaligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; }

}  // namespace

extern "C" size_t sv_lmhead_workspace_size(int N, int D, int V) {
  int a, b;
  size_t bytes;
  return lmhead_sizes(N, D, V, &a, &b, &bytes) ? bytes : 0;
}

extern "C" int sv_lmhead_stats(const void* hidden, const void* weight, const int32_t* tokens,
                               int N, int D, int V, float temperature, double* row_max,
                               double* lse, float* at, void* workspace, size_t workspace_bytes,
                               void* stream) {
  int n_mt, n_nt;
  size_t need;
  if (!lmhead_sizes(N, D, V, &n_mt, &n_nt, &need)) return SV_ERR_SHAPE;
  if (!std::isfinite(temperature) || !(temperature > 0.0f)) return SV_ERR_TEMPERATURE;
  if (N == 0) return SV_OK;
  if (!hidden || !weight || !tokens || !row_max || !lse || !at || !workspace) return SV_ERR_NULL;
  if (misaligned(hidden, 16) || misaligned(weight, 16) || misaligned(tokens, 4) ||
      misaligned(row_max, 8) || misaligned(lse, 8) || misaligned(at, 4) ||
      misaligned(workspace, 256))
    return SV_ERR_ALIGN;
  if (workspace_bytes < need) return SV_ERR_WORKSPACE;
  CUtensorMap mh, mw;
  if (!make_map(&mh, hidden, N, D, kBM) || !make_map(&mw, weight, V, D, kBN)) return SV_ERR_CUDA;
  // The kernel's shared-memory size is raised once per device (an attribute
  // of the function in the device's context).
  static std::mutex attr_mu;
  static bool attr_set[64] = {};
  static int sm_count[64] = {};
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= 64) return SV_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(attr_mu);
    if (!attr_set[device]) {
      if (cudaFuncSetAttribute(lmhead_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes) != cudaSuccess ||
          cudaDeviceGetAttribute(&sm_count[device], cudaDevAttrMultiProcessorCount, device) !=
              cudaSuccess || sm_count[device] < 1)
        return SV_ERR_CUDA;
      attr_set[device] = true;
    }
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  Args a{};
  a.tokens = tokens;
  a.N = N;
  a.D = D;
  a.V = V;
  a.n_mt = n_mt;
  a.n_nt = n_nt;
  a.nk = (D + kBK - 1) / kBK;
  a.n_tiles = n_mt * n_nt;
  const double T = (double)temperature;
  a.c2 = (float)(1.4426950408889634074 / T);
  a.part = reinterpret_cast<float2*>(ws + 256);
  a.at = at;
  a.status = reinterpret_cast<unsigned*>(ws);
  if (cudaMemsetAsync(ws, 0, 4, st) != cudaSuccess) return SV_ERR_CUDA;
  lmhead_kernel<<<(unsigned)std::min(a.n_tiles, sm_count[device]), kThreads, kSmemBytes, st>>>(
      mh, mw, a);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  const int rows_per_cta = 8;
  lmhead_combine_kernel<<<(unsigned)((N + rows_per_cta - 1) / rows_per_cta), 32 * rows_per_cta,
                          0, st>>>(a, 1.0 / T, row_max, lse);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
