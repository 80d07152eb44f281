// vm_cube.cu — the CUBE kernel type of the DVM interpreter (sm_103a): the MatMul tile
// op on the 5th-generation tensor cores, followed by the program's element-wise
// epilogue.  This is the "matmul + elemwise" fusion pattern of the DVM review page
// (section 5.2) and the cube flow of its execution model (section 3.2, Fig 3); the
// MindSpore DVM summary (section 3.3) describes the same cube-vector fusion.
//
// One persistent CTA per SM runs body_tile tiles (section 4.4).  Which tiles a core
// takes does not change any result, so the kernel deals them round-robin (tiles c,
// c + grid, c + 2*grid, ...): the tiles in flight at one time are neighbours in the
// row-major tile grid and share their A and W blocks in L2, where contiguous ranges
// would spread the working set over the whole of A.  A tile is 128 x t_N outputs.  Roles:
//   warp 0, one lane   TMA producer: the A [128 x 64] and W [t_N x 64] k-blocks of each
//                      tile go into a ring of shared-memory stages with the 128-byte
//                      swizzle, completion counted on the stage's mbarrier;
//   warp 1, one lane   MMA issuer: per k-block, four tcgen05.mma.kind::f16 (bf16 x bf16,
//                      fp32 accumulate, K = 16 each) into a TMEM accumulator; the stage is
//                      released by tcgen05.commit when those MMAs have read it.  The
//                      accumulator is double-buffered in TMEM so the epilogue of one tile
//                      overlaps the MMAs of the next.  Warp 1 owns the TMEM allocation;
//   warps 2..5         epilogue: thread i of the four warps owns accumulator row i (TMEM
//                      lane i), reads it 32 columns at a time with tcgen05.ld and runs the
//                      body's element-wise words (loads of bias/other operands, the
//                      element-wise ops, the bf16 cast, the store) on those 32 values in
//                      registers.
// Every wait is bounded by a time limit.  On expiry the CTA records DVM_E_TIMEOUT in the
// status word and raises its abort flag; each role stops, the producer waits (bounded)
// for its copies in flight, the issuer waits (bounded) for its MMAs, TMEM is freed and
// the CTA returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "dvm_internal.h"
#include "vm_common.cuh"

namespace dvm {

namespace {

constexpr int kCubeThreads = 192;
constexpr int kBM = 128;   // tile rows (MMA M)
constexpr int kBK = 64;    // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int kUK = 16;    // K of one tcgen05.mma.kind::f16

struct CubeParams {
  CUtensorMap tmA;         // A [M, K], box {64, min(128, M rounded up to 8)}
  CUtensorMap tmW;         // W as [N, K] (K contiguous), box {64, t_N}
  alignas(16) uint8_t image[kMaxImage];
  void* ptrs[kMaxBind];
  int32_t* status;
  float* ws;               // K-split partial tiles: [output tile][split][128 rows][t_N] fp32
  int* ws_count;           // K-split arrivals per output tile (zero between launches)
  unsigned long long timeout_ns;
  uint32_t image_len;
};

// shared-memory layout after the 1024-byte aligned ring
struct CubeCtl {
  uint64_t full[kCubeMaxStages];
  uint64_t empty[kCubeMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t esync;   // the epilogue warps' barrier (bounded waits)
  uint32_t tmem_base;
  int abort;
  int n_ep;         // decoded epilogue micro-ops
  int ep_last[2];   // this CTA completes the output tile of its K-split (by tile parity)
};
constexpr int kCubeCtlBytes = 1024;
static_assert(sizeof(CubeCtl) <= kCubeCtlBytes, "control block");

// ------------------------------------------------------------ TMA, tcgen05 --
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tc_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accum)
      : "memory");
}
// the mbarrier's arrival fires when every tcgen05 op this thread issued so far is done
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane; the wait is in the same
// statement so no use of the registers can be scheduled before the data is there.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand tile stored as rows of 128 bytes
// (64 bf16 along K) with the 128-byte swizzle, 8-row groups 1024 bytes apart: start
// address >> 4 in bits 0-13, leading-dimension offset (unused for this layout) 16 B in
// bits 16-29, stride-dimension offset 1024 B in bits 32-45, descriptor version 1 in
// bits 46-47, base offset 0 (tiles are 1024-byte aligned), swizzle mode 2 (128-byte) in
// bits 61-63.  Moving along K by 16 elements adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of tcgen05.mma.kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t mma_idesc(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// bounded wait without the suspend hint, for the roles on the MMA critical path (the
// producer and the MMA issuer): a tight poll, with the clock and abort checked every 64
// polls
__device__ __forceinline__ bool mbar_spin(uint64_t* bar, uint32_t parity, const DevStatus& st, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; i++)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > st.limit_ns) {
      set_status(st.word, -100 /* DVM_E_TIMEOUT */);
      *abort = 1;
      return false;
    }
  }
}

// barrier of the four epilogue warps on an mbarrier of 128 arrivals: a bounded wait, so a
// warp that left its loop on abort cannot hold the others forever
__device__ __forceinline__ bool ep_sync(uint64_t* bar, uint32_t& ph, const DevStatus& st, volatile int* abort) {
  mbar_arrive(bar);
  const bool ok = mbar_wait(bar, ph, st, abort);
  ph ^= 1u;
  return ok;
}

// bounded wait that ignores the abort flag (draining copies and MMAs before exit)
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait_sleep(bar, parity, 20000u))
    if (globaltimer() - t0 > limit_ns) return false;
  return true;
}

// ------------------------------------------------------------- epilogue ops --
__device__ __forceinline__ float ld_elem(const uint8_t* base, int dt, int64_t i) {
  if (dt == DT_F32) return reinterpret_cast<const float*>(base)[i];
  if (dt == DT_BF16) return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(base)[i] << 16);
  return (float)base[i];
}
__device__ __forceinline__ void st_elem(uint8_t* base, int dt, int64_t i, float v) {
  if (dt == DT_F32) reinterpret_cast<float*>(base)[i] = v;
  else if (dt == DT_BF16) reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  else base[i] = (uint8_t)(v != 0.f ? 1 : 0);
}

// 32 values of (row m, columns n0..n0+31) of a bound tensor; columns >= n0+nvalid read 0
__device__ __forceinline__ void ep_load(float (&x)[32], int dt, int64_t vs0, int64_t vs1, const uint8_t* base, int m,
                                        int n0, int nvalid) {
  const int esz = dtype_size(dt);
  if (vs1 == 0) {  // one value per row
    const float v = ld_elem(base, dt, (int64_t)m * vs0);
#pragma unroll
    for (int i = 0; i < 32; i++) x[i] = v;
    return;
  }
  const int64_t off = (int64_t)m * vs0 + (int64_t)n0 * vs1;
  const uint8_t* p = base + off * esz;
  if (vs1 == 1 && nvalid == 32 && ((uintptr_t)p & 15) == 0) {
    if (dt == DT_F32) {
#pragma unroll
      for (int q = 0; q < 8; q++) {
        const float4 v = reinterpret_cast<const float4*>(p)[q];
        x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
      }
    } else if (dt == DT_BF16) {
#pragma unroll
      for (int q = 0; q < 4; q++) {
        const uint4 v = reinterpret_cast<const uint4*>(p)[q];
        x[8 * q + 0] = bf16lo(v.x); x[8 * q + 1] = bf16hi(v.x);
        x[8 * q + 2] = bf16lo(v.y); x[8 * q + 3] = bf16hi(v.y);
        x[8 * q + 4] = bf16lo(v.z); x[8 * q + 5] = bf16hi(v.z);
        x[8 * q + 6] = bf16lo(v.w); x[8 * q + 7] = bf16hi(v.w);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 2; q++) {
        const uint4 v = reinterpret_cast<const uint4*>(p)[q];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 16; j++) x[16 * q + j] = (float)((w[j >> 2] >> (8 * (j & 3))) & 0xffu);
      }
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 32; i++) x[i] = i < nvalid ? ld_elem(base, dt, off + (int64_t)i * vs1) : 0.f;
}

__device__ __forceinline__ void ep_store(const float (&x)[32], int dt, int64_t vs0, int64_t vs1, uint8_t* base, int m,
                                         int n0, int nvalid) {
  const int esz = dtype_size(dt);
  const int64_t off = (int64_t)m * vs0 + (int64_t)n0 * vs1;
  uint8_t* p = base + off * esz;
  if (vs1 == 1 && nvalid == 32 && ((uintptr_t)p & 15) == 0) {
    if (dt == DT_F32) {
#pragma unroll
      for (int q = 0; q < 8; q++)
        reinterpret_cast<float4*>(p)[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    } else if (dt == DT_BF16) {
#pragma unroll
      for (int q = 0; q < 4; q++)
        reinterpret_cast<uint4*>(p)[q] =
            make_uint4(pack_bf16(x[8 * q], x[8 * q + 1]), pack_bf16(x[8 * q + 2], x[8 * q + 3]),
                       pack_bf16(x[8 * q + 4], x[8 * q + 5]), pack_bf16(x[8 * q + 6], x[8 * q + 7]));
    } else {
#pragma unroll
      for (int q = 0; q < 2; q++) {
        uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 16; j++) w[j >> 2] |= (x[16 * q + j] != 0.f ? 1u : 0u) << (8 * (j & 3));
        reinterpret_cast<uint4*>(p)[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 32; i++)
    if (i < nvalid) st_elem(base, dt, off + (int64_t)i * vs1, x[i]);
}

__device__ __forceinline__ float ep_unary(int op, float x) {
  switch (op) {
    case OP_SQRT: return sqrtf(x);
    case OP_ABS: return fabsf(x);
    case OP_LOG: return logf(x);
    case OP_EXP: return expf(x);
    case OP_ROUND: return rintf(x);
    case OP_FLOOR: return floorf(x);
    case OP_ISFIN: return isfinite(x) ? 1.f : 0.f;
    case OP_NEG: return -x;
    case OP_RSQRT: return 1.0f / sqrtf(x);
    case OP_RECIP: return 1.0f / x;
    case OP_SILU: return x / (1.0f + expf(-x));
    default: return round_bf16(x);  // OP_CASTBF
  }
}
__device__ __forceinline__ float ep_binary(int op, float a, float b) {
  switch (op) {
    case OP_ADD: return a + b;
    case OP_SUB: return a - b;
    case OP_MUL: return a * b;
    case OP_DIV: return a / b;
    case OP_MAX: return vmax(a, b);
    case OP_MIN: return vmin(a, b);
    default: return powf(a, b);
  }
}

template <int OP>
__device__ __forceinline__ void ep_bin_loop(float (&acc)[32], const float (&x)[32], bool rev) {
  if (rev) {
#pragma unroll
    for (int i = 0; i < 32; i++) acc[i] = ep_binary(OP, x[i], acc[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 32; i++) acc[i] = ep_binary(OP, acc[i], x[i]);
  }
}
template <int OP>
__device__ __forceinline__ void ep_un_loop(float (&acc)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i++) acc[i] = ep_unary(OP, acc[i]);
}

__device__ __forceinline__ void sel_slot(float (&x)[32], int k, const float (&acc)[32], const float (&s1)[32],
                                         const float (&s2)[32]) {
  if (k == 1) {
#pragma unroll
    for (int i = 0; i < 32; i++) x[i] = s1[i];
  } else if (k == 2) {
#pragma unroll
    for (int i = 0; i < 32; i++) x[i] = s2[i];
  } else {
#pragma unroll
    for (int i = 0; i < 32; i++) x[i] = acc[i];
  }
}
__device__ __forceinline__ void put_slot(const float (&x)[32], int k, float (&acc)[32], float (&s1)[32], float (&s2)[32]) {
  if (k == 1) {
#pragma unroll
    for (int i = 0; i < 32; i++) s1[i] = x[i];
  } else if (k == 2) {
#pragma unroll
    for (int i = 0; i < 32; i++) s2[i] = x[i];
  } else {
#pragma unroll
    for (int i = 0; i < 32; i++) acc[i] = x[i];
  }
}

// ---- the epilogue, decoded once per CTA ---------------------------------------------
// The epilogue words are decoded into micro-ops with their tensors resolved (base
// pointer, strides, element type), and neighbours are fused so that a 32-column chunk
// costs fewer dispatches: a load into a slot followed by a light op reading that slot
// (when no later word reads the slot), a CASTBF followed by a store, and ops with an
// immediate operand get their own handlers.
enum EpHandler : uint8_t {
  E_LD, E_ST, E_STB, E_MOV, E_BIN, E_OPLD_ADD, E_OPLD_SUB, E_OPLD_RSUB, E_OPLD_MUL,
  E_ADDI, E_SUBI, E_RSUBI, E_MULI, E_ABS, E_NEG, E_CASTBF, E_UN, E_NOP
};
struct alignas(16) EpOp {
  const uint8_t* base;  // tensor base (loads, stores)
  int64_t vs0, vs1;     // element strides of the tensor over (row, column)
  float imm;
  uint8_t h, a, b, fl;
  uint8_t dt, op, pad0, pad1;
  uint32_t pad2;
};
static_assert(sizeof(EpOp) == 48, "epilogue micro-op");
constexpr int kMaxEpOps = kMaxInstr;  // an epilogue never has more words than a body

__device__ __forceinline__ bool ep_reads_slot(const Instr& w, int k) {
  if (w.op == OP_MOV) return w.b == k;
  if (w.op >= OP_ADD && w.op <= OP_POW) return !(w.flags & CF_IMM) && w.a == k;
  return false;
}
__device__ __forceinline__ bool ep_slot_live_after(const Instr* w, int n, int i, int k) {
  for (int j = i + 1; j < n; j++) {
    if (ep_reads_slot(w[j], k)) return true;
    if ((w[j].op == OP_LD || w[j].op == OP_MOV) && w[j].a == k) return false;
  }
  return false;
}

// decode (one thread); returns the number of micro-ops
__device__ __forceinline__ int ep_decode(const Instr* w, int n, const TensRec* tens, void* const* ptrs, EpOp* E) {
  int m = 0;
  for (int i = 0; i < n && m < kMaxEpOps; i++) {
    const Instr I = w[i];
    EpOp e;
    e.base = nullptr;
    e.vs0 = e.vs1 = 0;
    e.imm = __uint_as_float(I.imm);
    e.h = E_NOP;
    e.a = I.a;
    e.b = I.b;
    e.fl = I.flags;
    e.dt = 0;
    e.op = I.op;
    const bool imm = I.flags & CF_IMM, rev = I.flags & CF_REV;
    switch (I.op) {
      case OP_LD: {
        const TensRec& t = tens[I.b];
        e.base = static_cast<const uint8_t*>(ptrs[t.binding]);
        e.vs0 = t.vs[0];
        e.vs1 = t.vs[1];
        e.dt = t.dtype;
        e.h = E_LD;
        if (I.a != 0 && i + 1 < n) {
          const Instr x = w[i + 1];
          if ((x.op == OP_ADD || x.op == OP_SUB || x.op == OP_MUL) && !(x.flags & CF_IMM) && x.a == I.a &&
              !ep_slot_live_after(w, n, i + 1, I.a)) {
            e.h = x.op == OP_ADD ? E_OPLD_ADD : x.op == OP_MUL ? E_OPLD_MUL : (x.flags & CF_REV) ? E_OPLD_RSUB : E_OPLD_SUB;
            i++;
          }
        }
        break;
      }
      case OP_ST: {
        const TensRec& t = tens[I.a];
        e.base = static_cast<const uint8_t*>(ptrs[t.binding]);
        e.vs0 = t.vs[0];
        e.vs1 = t.vs[1];
        e.dt = t.dtype;
        e.h = E_ST;
        break;
      }
      case OP_CASTBF:
        e.h = E_CASTBF;
        if (i + 1 < n && w[i + 1].op == OP_ST) {
          const TensRec& t = tens[w[i + 1].a];
          e.base = static_cast<const uint8_t*>(ptrs[t.binding]);
          e.vs0 = t.vs[0];
          e.vs1 = t.vs[1];
          e.dt = t.dtype;
          e.h = E_STB;
          i++;
        }
        break;
      case OP_MOV: e.h = E_MOV; break;
      case OP_ADD: case OP_SUB: case OP_MUL:
        if (imm) e.h = I.op == OP_ADD ? E_ADDI : I.op == OP_MUL ? E_MULI : rev ? E_RSUBI : E_SUBI;
        else e.h = E_BIN;
        break;
      case OP_DIV: case OP_MAX: case OP_MIN: case OP_POW: e.h = E_BIN; break;
      case OP_ABS: e.h = E_ABS; break;
      case OP_NEG: e.h = E_NEG; break;
      case OP_BCAST: case OP_WAIT: case OP_REL: e.h = E_NOP; break;
      default: e.h = E_UN; break;
    }
    E[m++] = e;
  }
  return m;
}

// Run the epilogue micro-ops on 32 accumulator values of row m (valid when m < M),
// columns n0..n0+nvalid-1.  Micro-ops are warp-uniform; loads and stores are skipped for
// rows outside the output.
__device__ void run_epilogue(const EpOp* E, int ne, float (&acc)[32], int m, bool row_ok, int n0, int nvalid) {
  float s1[32], s2[32], x[32];
#pragma unroll
  for (int i = 0; i < 32; i++) s1[i] = s2[i] = 0.f;
  for (int k = 0; k < ne; k++) {
    const EpOp e = E[k];
    switch (e.h) {
      case E_LD:
        if (row_ok) ep_load(x, e.dt, e.vs0, e.vs1, e.base, m, n0, nvalid);
        else {
#pragma unroll
          for (int i = 0; i < 32; i++) x[i] = 0.f;
        }
        put_slot(x, e.a, acc, s1, s2);
        break;
      case E_OPLD_ADD: case E_OPLD_SUB: case E_OPLD_RSUB: case E_OPLD_MUL:
        if (row_ok) ep_load(x, e.dt, e.vs0, e.vs1, e.base, m, n0, nvalid);
        else {
#pragma unroll
          for (int i = 0; i < 32; i++) x[i] = 0.f;
        }
        if (e.h == E_OPLD_ADD) {
#pragma unroll
          for (int i = 0; i < 32; i++) acc[i] = acc[i] + x[i];
        } else if (e.h == E_OPLD_MUL) {
#pragma unroll
          for (int i = 0; i < 32; i++) acc[i] = acc[i] * x[i];
        } else if (e.h == E_OPLD_SUB) {
#pragma unroll
          for (int i = 0; i < 32; i++) acc[i] = acc[i] - x[i];
        } else {
#pragma unroll
          for (int i = 0; i < 32; i++) acc[i] = x[i] - acc[i];
        }
        break;
      case E_ST:
        if (row_ok) ep_store(acc, e.dt, e.vs0, e.vs1, const_cast<uint8_t*>(e.base), m, n0, nvalid);
        break;
      case E_STB:
#pragma unroll
        for (int i = 0; i < 32; i++) acc[i] = round_bf16(acc[i]);
        if (row_ok) ep_store(acc, e.dt, e.vs0, e.vs1, const_cast<uint8_t*>(e.base), m, n0, nvalid);
        break;
      case E_MOV:
        sel_slot(x, e.b, acc, s1, s2);
        put_slot(x, e.a, acc, s1, s2);
        break;
      case E_ADDI:
#pragma unroll
        for (int i = 0; i < 32; i++) acc[i] = acc[i] + e.imm;
        break;
      case E_SUBI:
#pragma unroll
        for (int i = 0; i < 32; i++) acc[i] = acc[i] - e.imm;
        break;
      case E_RSUBI:
#pragma unroll
        for (int i = 0; i < 32; i++) acc[i] = e.imm - acc[i];
        break;
      case E_MULI:
#pragma unroll
        for (int i = 0; i < 32; i++) acc[i] = acc[i] * e.imm;
        break;
      case E_ABS:
#pragma unroll
        for (int i = 0; i < 32; i++) acc[i] = fabsf(acc[i]);
        break;
      case E_NEG:
#pragma unroll
        for (int i = 0; i < 32; i++) acc[i] = -acc[i];
        break;
      case E_CASTBF:
#pragma unroll
        for (int i = 0; i < 32; i++) acc[i] = round_bf16(acc[i]);
        break;
      case E_BIN: {
        if (e.fl & CF_IMM) {
#pragma unroll
          for (int i = 0; i < 32; i++) x[i] = e.imm;
        } else {
          sel_slot(x, e.a, acc, s1, s2);
        }
        const bool rev = (e.fl & CF_REV) != 0;
        switch (e.op) {
          case OP_ADD: ep_bin_loop<OP_ADD>(acc, x, rev); break;
          case OP_SUB: ep_bin_loop<OP_SUB>(acc, x, rev); break;
          case OP_MUL: ep_bin_loop<OP_MUL>(acc, x, rev); break;
          case OP_DIV: ep_bin_loop<OP_DIV>(acc, x, rev); break;
          case OP_MAX: ep_bin_loop<OP_MAX>(acc, x, rev); break;
          case OP_MIN: ep_bin_loop<OP_MIN>(acc, x, rev); break;
          default: ep_bin_loop<OP_POW>(acc, x, rev); break;
        }
        break;
      }
      case E_UN:
        switch (e.op) {
          case OP_SQRT: ep_un_loop<OP_SQRT>(acc); break;
          case OP_LOG: ep_un_loop<OP_LOG>(acc); break;
          case OP_EXP: ep_un_loop<OP_EXP>(acc); break;
          case OP_ROUND: ep_un_loop<OP_ROUND>(acc); break;
          case OP_FLOOR: ep_un_loop<OP_FLOOR>(acc); break;
          case OP_ISFIN: ep_un_loop<OP_ISFIN>(acc); break;
          case OP_RSQRT: ep_un_loop<OP_RSQRT>(acc); break;
          case OP_RECIP: ep_un_loop<OP_RECIP>(acc); break;
          case OP_SILU: ep_un_loop<OP_SILU>(acc); break;
          default: break;  // the validator admits nothing else in a CUBE body
        }
        break;
      default:
        break;
    }
  }
}

// ------------------------------------------------------------------ kernel --
__global__ void __launch_bounds__(kCubeThreads, 1) vm_cube_kernel(const __grid_constant__ CubeParams P) {
  const Header* H = reinterpret_cast<const Header*>(P.image);
  const int cta = blockIdx.x;
  const int nblk = (int)H->block_dim;
  const int step = (int)gridDim.x;
  const int lo = cta;     // this CTA's tiles: lo, lo + step, ... < nblk
  const int hi = nblk;
  if (lo >= hi) return;  // uniform over the CTA: nothing to do, nothing allocated

  extern __shared__ uint8_t cube_smem_raw[];
  const uint32_t raw = smem_u32(cube_smem_raw);
  uint8_t* smem = cube_smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int S = H->n_stages;
  const uint32_t stage_bytes = H->stage_bytes;
  CubeCtl* C = reinterpret_cast<CubeCtl*>(smem + (size_t)S * stage_bytes);
  EpOp* eops = reinterpret_cast<EpOp*>(smem + (size_t)S * stage_bytes + kCubeCtlBytes);
  uint8_t* img = smem + (size_t)S * stage_bytes + kCubeCtlBytes + kMaxEpOps * sizeof(EpOp);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // image -> shared memory (the epilogue decodes its words from there)
  for (uint32_t i = tid * 16; i < P.image_len; i += kCubeThreads * 16)
    *reinterpret_cast<uint4*>(img + i) = *reinterpret_cast<const uint4*>(P.image + i);
  if (tid == 0) {
    for (int s = 0; s < S; s++) {
      mbar_init(&C->full[s], 1);
      mbar_init(&C->empty[s], 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&C->tfull[b], 1);
      mbar_init(&C->tempty[b], 128);
    }
    mbar_init(&C->drain, 1);
    mbar_init(&C->esync, 128);
    C->abort = 0;
    fence_mbar_init();
  }
  const ProgRec* pr = reinterpret_cast<const ProgRec*>(P.image + sizeof(Header));
  const int M = (int)pr->n[0], N = (int)pr->n[1], K = (int)pr->K;
  const int BN = (int)pr->t[1];
  const int tiles_n = (N + BN - 1) / BN;
  // a work unit is one K-split of one output tile: unit = tile * ks + split
  const int TK = (int)pr->t[2];
  const int ks = (K + TK - 1) / TK;
  // A's TMA box is min(128, M rounded up to 8) rows, and a stage holds only those rows
  // followed by the W block: an instance with fewer than 128 rows copies no zero fill and
  // fits more stages in the ring.  The MMA still reads a 128-row A operand; its rows
  // beyond the box read whatever follows in shared memory (W, later stages, the control
  // block, or the slack the launch allocates past them) and feed only accumulator rows
  // that the epilogue never stores.
  const uint32_t a_box_bytes = (uint32_t)min(kBM, (M + 7) & ~7) * kBK * 2;
  // two accumulators of BN columns, each starting on a multiple of 32 columns so that
  // the epilogue's 32-column reads stay inside the accumulator they belong to
  const int BNp = (BN + 31) & ~31;
  uint32_t ncols = 32;
  while (ncols < 2u * (uint32_t)BNp) ncols <<= 1;
  if (warp == 1) {
    tc_alloc(smem_u32(&C->tmem_base), ncols);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C->tmem_base;
  const DevStatus st{P.status, P.timeout_ns};
  volatile int* abort = &C->abort;
  const uint32_t ring = smem_u32(smem);

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer --
    if (lane == 0) {
      tma_prefetch_map(&P.tmA);
      tma_prefetch_map(&P.tmW);
      // stage index, phase and destination advance incrementally: this thread issues a
      // stage every few hundred cycles at the peak MMA rate, so the loop carries no
      // division and no reload of anything but the barrier word
      const uint32_t tx_bytes = a_box_bytes + (uint32_t)BN * kBK * 2;
      int it = 0, s = 0;
      uint32_t ph = 0, a_dst = ring;
      bool ok = true;
      for (int tau = lo; tau < hi && ok && !*abort; tau += step) {
        const int tile = tau / ks, kk = tau - tile * ks;
        const int tm = tile / tiles_n, tn = tile - tm * tiles_n;
        const int ya = tm * kBM, yw = tn * BN;
        const int k1 = min(K, (kk + 1) * TK);
        for (int kx = kk * TK; kx < k1; kx += kBK, it++) {
          if (!mbar_spin(&C->empty[s], ph ^ 1u, st, abort)) { ok = false; break; }
          mbar_arrive_expect_tx(&C->full[s], tx_bytes);
          tma_load_2d(a_dst, &P.tmA, kx, ya, &C->full[s]);
          tma_load_2d(a_dst + a_box_bytes, &P.tmW, kx, yw, &C->full[s]);
          a_dst += stage_bytes;
          if (++s == S) { s = 0; ph ^= 1u; a_dst = ring; }
        }
      }
      // copies still in flight land before the CTA may exit (normally all have landed)
      for (int j = it > S ? it - S : 0; j < it; j++)
        if (!mbar_drain(&C->full[j % S], (uint32_t)(j / S) & 1u, st.limit_ns)) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer --
    if (lane == 0) {
      const uint32_t idesc = mma_idesc(kBM, BN);
      // the descriptors of stage 0; a stage further on adds stage_bytes >> 4 to the start
      // address field (shared addresses stay below 2^18, so the field cannot carry)
      const uint64_t da0 = sw128_desc(ring), db0 = sw128_desc(ring + a_box_bytes);
      const uint64_t dstep = stage_bytes >> 4;
      int jt = 0, s = 0;
      uint32_t ph = 0;
      uint64_t da = da0, db = db0;
      bool issued = false, ok = true;
      for (int tau = lo; tau < hi && ok && !*abort; tau += step, jt++) {
        const int b = jt & 1;
        const uint32_t use = (uint32_t)(jt >> 1);
        if (!mbar_spin(&C->tempty[b], (use & 1u) ^ 1u, st, abort)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * BNp);
        const int kk = tau % ks;
        const int nkb_u = (min(K, (kk + 1) * TK) - kk * TK + kBK - 1) / kBK;
        uint32_t acc = 0;
        for (int kb = 0; kb < nkb_u; kb++) {
          if (!mbar_spin(&C->full[s], ph, st, abort)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kBK / kUK; k++) {
            tc_mma(d, da + (uint64_t)(k * 2), db + (uint64_t)(k * 2), idesc, acc);
            acc = 1u;
          }
          issued = true;
          tc_commit(&C->empty[s]);
          da += dstep;
          db += dstep;
          if (++s == S) { s = 0; ph ^= 1u; da = da0; db = db0; }
        }
        if (!ok) break;
        tc_commit(&C->tfull[b]);
      }
      if (issued) {  // every MMA of this CTA has finished before TMEM is freed
        tc_commit(&C->drain);
        mbar_drain(&C->drain, 0, st.limit_ns);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue --
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;          // accumulator row owned by this thread
    const ProgRec* spr = reinterpret_cast<const ProgRec*>(img + sizeof(Header));
    const Instr* body = reinterpret_cast<const Instr*>(img + spr->body_off);
    const TensRec* tens = reinterpret_cast<const TensRec*>(img + spr->tens_off);
    const int n_epi = (int)body[0].imm - 1;  // words after the MMA word
    // decode the epilogue once (first epilogue thread), then sync the epilogue warps
    if (threadIdx.x == 64) C->n_ep = ep_decode(body + 2, n_epi, tens, P.ptrs, eops);
    named_bar(2, 128);
    const int ne = C->n_ep;
    int jt = 0;
    uint32_t eph = 0;
    for (int tau = lo; tau < hi; tau += step, jt++) {
      const int b = jt & 1;
      if (!mbar_wait(&C->tfull[b], (uint32_t)(jt >> 1) & 1u, st, abort)) break;
      tc_fence_after();
      const int tile = tau / ks;
      const int tm = tile / tiles_n, tn = tile - tm * tiles_n;
      const int m = tm * kBM + row;
      const bool row_ok = m < M;
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BNp);
      if (ks == 1) {
        for (int c = 0; c < BN; c += 32) {
          const int n0 = tn * BN + c;
          if (n0 >= N) break;  // warp-uniform
          float acc[32];
          tc_ld32(tacc + (uint32_t)c, acc);
          run_epilogue(eops, ne, acc, m, row_ok, n0, min(min(32, BN - c), N - n0));
        }
        tc_fence_before();
        mbar_arrive(&C->tempty[b]);
        continue;
      }
      // K-split: store this split's fp32 partial rows, count the split in; the CTA that
      // brings the count to ks sums the partials in split order and runs the epilogue
      float* own = P.ws + ((size_t)tau * kBM + row) * BN;
      for (int c = 0; c < BN; c += 32) {
        float acc[32];
        tc_ld32(tacc + (uint32_t)c, acc);
        if (row_ok) {
          float4* d4 = reinterpret_cast<float4*>(own + c);
#pragma unroll
          for (int i = 0; i < 8; i++)
            if (c + 4 * i < BN) d4[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&C->tempty[b]);
      __threadfence();
      if (!ep_sync(&C->esync, eph, st, abort)) break;
      if (threadIdx.x == 64) {
        const int old = atomicAdd(P.ws_count + tile, 1);
        const int last = old == ks - 1 ? 1 : 0;
        if (last) P.ws_count[tile] = 0;  // every split of this launch has counted in
        C->ep_last[jt & 1] = last;
        __threadfence();
      }
      if (!ep_sync(&C->esync, eph, st, abort)) break;
      if (!*reinterpret_cast<volatile int*>(&C->ep_last[jt & 1])) continue;
      __threadfence();
      // this CTA completes the tile.  (1) the 128 epilogue threads sum the splits' float4
      // columns in split order, in place over split 0; (2) they run the epilogue over
      // (row, 32-column) chunks of the sum.  Both spread the tile over all threads, so a
      // tile of few rows is summed as fast as a full one per byte.
      const int et = threadIdx.x - 64;
      const int rows_v = min(kBM, M - tm * kBM), cols_v = min(BN, N - tn * BN);
      float* part = P.ws + (size_t)tile * ks * kBM * BN;
      const size_t sstride = (size_t)kBM * BN / 4;  // float4s between splits
      const int nf4 = (cols_v + 3) / 4, n_sum = rows_v * nf4;
      constexpr int U = 4;
      for (int i0 = et; i0 < n_sum; i0 += 128 * U) {
        float4 a[U];
        float4* p4[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
          const int i = min(i0 + u * 128, n_sum - 1);
          const int r = i / nf4;
          p4[u] = reinterpret_cast<float4*>(part + (size_t)r * BN) + (i - r * nf4);
          a[u] = __ldcg(p4[u]);
        }
#pragma unroll 4
        for (int sp = 1; sp < ks; sp++) {
#pragma unroll
          for (int u = 0; u < U; u++) {
            const float4 v = __ldcg(p4[u] + sp * sstride);
            a[u].x += v.x;
            a[u].y += v.y;
            a[u].z += v.z;
            a[u].w += v.w;
          }
        }
#pragma unroll
        for (int u = 0; u < U; u++)
          if (i0 + u * 128 < n_sum) __stcg(p4[u], a[u]);
      }
      if (!ep_sync(&C->esync, eph, st, abort)) break;
      const int nch = (cols_v + 31) / 32;
      for (int i = et; i < rows_v * nch; i += 128) {
        const int r = i / nch, c = (i - r * nch) * 32;
        const float4* s4 = reinterpret_cast<const float4*>(part + (size_t)r * BN + c);
        float acc[32];
#pragma unroll
        for (int q4 = 0; q4 < 8; q4++) {
          const float4 v = c + 4 * q4 < BN ? __ldcg(s4 + q4) : make_float4(0.f, 0.f, 0.f, 0.f);
          acc[4 * q4] = v.x;
          acc[4 * q4 + 1] = v.y;
          acc[4 * q4 + 2] = v.z;
          acc[4 * q4 + 3] = v.w;
        }
        run_epilogue(eops, ne, acc, tm * kBM + r, true, tn * BN + c, min(32, cols_v - c));
      }
      if (!ep_sync(&C->esync, eph, st, abort)) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc(tmem, ncols);
  }
}

// ------------------------------------------------------------------- host --
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(char* msg, size_t cap) {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!fn) std::snprintf(msg, cap, "cuTensorMapEncodeTiled is not available from the driver");
  return fn;
}

// 2-D bf16 tensor map: `rows` x `k` elements, row pitch `pitch_bytes`, box {64, box_rows}
bool make_map(EncodeTiledFn fn, CUtensorMap* map, void* base, uint64_t k, uint64_t rows, uint64_t pitch_bytes,
              uint32_t box_rows) {
  const cuuint64_t dims[2] = {k, rows};
  const cuuint64_t strides[1] = {pitch_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

int cube_launch(DeviceState* st, const uint8_t* image, size_t len, void* const* ptrs, int n, void* stream, char* msg,
                size_t cap) {
  Header h;
  std::memcpy(&h, image, sizeof h);
  ProgRec pr;
  std::memcpy(&pr, image + sizeof(Header), sizeof pr);
  Instr w0, w1;
  std::memcpy(&w0, image + pr.body_off, sizeof w0);
  std::memcpy(&w1, image + pr.body_off + sizeof(Instr), sizeof w1);
  if (h.n_progs != 1 || w0.op != OP_TILES || w1.op != OP_MMA) {
    std::snprintf(msg, cap, "a CUBE image holds one program whose tile body starts with MMA");
    return -5;
  }
  TensRec ta, tw;
  std::memcpy(&ta, image + pr.tens_off + w1.a * sizeof(TensRec), sizeof ta);
  std::memcpy(&tw, image + pr.tens_off + w1.b * sizeof(TensRec), sizeof tw);
  const uint64_t M = pr.n[0], N = pr.n[1], K = pr.K, BN = pr.t[1];
  const size_t ring = (size_t)h.n_stages * h.stage_bytes;
  const uint32_t a_rows = M >= (uint64_t)kBM ? (uint32_t)kBM : (uint32_t)((M + 7) / 8 * 8);
  if (ta.dtype != DT_BF16 || tw.dtype != DT_BF16 || ta.vs[1] != 1 || tw.vs[0] != 1 || h.n_stages < 2 ||
      h.n_stages > kCubeMaxStages || h.stage_bytes != (uint32_t)((a_rows + BN) * kBK * 2) ||
      ring > (size_t)kCubeRingBytes) {
    std::snprintf(msg, cap, "CUBE operands must be bf16 and K-contiguous with a valid stage ring");
    return -5;
  }
  // row pitches in bytes (a single row may have any stride: only row 0 is read)
  uint64_t pa = M == 1 ? (K * 2 + 15) / 16 * 16 : (uint64_t)ta.vs[0] * 2;
  uint64_t pw = N == 1 ? (K * 2 + 15) / 16 * 16 : (uint64_t)tw.vs[1] * 2;
  if (pa == 0 || pw == 0 || pa % 16 || pw % 16) {
    std::snprintf(msg, cap, "MatMul row pitches must be non-zero multiples of 16 bytes");
    return -5;
  }
  EncodeTiledFn fn = encode_fn(msg, cap);
  if (!fn) return -6;
  static thread_local CubeParams P;
  if (!make_map(fn, &P.tmA, ptrs[ta.binding], K, M, pa, a_rows) ||
      !make_map(fn, &P.tmW, ptrs[tw.binding], K, N, pw, (uint32_t)BN)) {
    std::snprintf(msg, cap, "cuTensorMapEncodeTiled rejected a MatMul operand");
    return -6;
  }
  std::memcpy(P.image, image, len);
  P.image_len = (uint32_t)((len + 15) / 16 * 16);
  for (int i = 0; i < n; i++) P.ptrs[i] = ptrs[i];
  P.status = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(st->scratch) + 8);
  P.timeout_ns = (unsigned long long)st->timeout_ms * 1000000ull;
  // K-split tiles: the context's workspace, allocated at its first K-split launch
  const uint64_t TK = pr.t[2];
  if ((K + TK - 1) / TK > 1 && !st->cube_ws) {
    const size_t bytes = (size_t)kCubeWsBytes + sizeof(int) * kCubeWsTiles;
    void* ws = nullptr;
    cudaError_t e = cudaMalloc(&ws, bytes);
    if (e == cudaSuccess) e = cudaMemset(static_cast<uint8_t*>(ws) + kCubeWsBytes, 0, sizeof(int) * kCubeWsTiles);
    if (e != cudaSuccess) {
      if (ws) cudaFree(ws);
      std::snprintf(msg, cap, "K-split workspace allocation failed: %s", cudaGetErrorString(e));
      return -6;
    }
    st->cube_ws = ws;
  }
  P.ws = static_cast<float*>(st->cube_ws);
  P.ws_count = st->cube_ws ? reinterpret_cast<int*>(static_cast<uint8_t*>(st->cube_ws) + kCubeWsBytes) : nullptr;
  // the last stage's 128-row A operand may reach (128 - a_rows) rows of 128 bytes past its
  // own A box and W block: the allocation covers that reach whatever follows the ring
  const size_t tail = (size_t)kCubeCtlBytes + kMaxEpOps * sizeof(EpOp) + P.image_len;
  const size_t reach = (size_t)(kBM - a_rows) * kBK * 2;
  const size_t over = reach > BN * kBK * 2 ? reach - BN * kBK * 2 : 0;
  const size_t smem = 1024 + ring + (over > tail ? over : tail);
  if ((int)smem > st->max_smem_optin) {
    std::snprintf(msg, cap, "CUBE shared memory %zu exceeds the device limit %d", smem, st->max_smem_optin);
    return -8;
  }
  static thread_local int attr_dev = -1;
  if (attr_dev != st->device) {
    cudaError_t e = cudaFuncSetAttribute(vm_cube_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, st->max_smem_optin);
    if (e != cudaSuccess) {
      std::snprintf(msg, cap, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      return -6;
    }
    attr_dev = st->device;
  }
  vm_cube_kernel<<<h.grid, kCubeThreads, smem, static_cast<cudaStream_t>(stream)>>>(P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    std::snprintf(msg, cap, "CUBE launch: %s", cudaGetErrorString(e));
    return -6;
  }
  st->launches++;
  return 0;
}

}  // namespace dvm
