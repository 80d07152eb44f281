// vm_vec.cuh — the persistent DVM interpreter for element-wise / reduce programs (VEC
// kernel type), sm_103a.
//
// Execution model (DVM review page, section 4.4 "virtual machine execution"): each CTA
// is one "AI core"; it computes its contiguous tile range [c*body_tile,
// min((c+1)*body_tile, block_dim)) and, for each tile, decodes the code body and calls
// the matching virtual-instruction function.  Decoding is warp-uniform from the image
// staged in shared memory.  Section 3.2's asynchronous flows map onto one CTA:
//   * DMA flow    -> one producer warp that streams tile rows from HBM into a ring of
//                    shared-memory stages with cp.async.bulk, signalled by mbarriers;
//   * vector flow -> 15 consumer warps that move a tile from its stage into registers
//                    (LD), run the element-wise chain in registers, reduce rows with
//                    warp shuffles, and store straight from registers to HBM (ST);
//   * the WAIT / REL words the encoder inserts are the syncs between the two flows.
// Registers follow an accumulator machine: ACC plus 2 slots of REG fp32 values per
// thread; every instruction reads ACC and at most one slot, so slot selection is a
// uniform switch with the computation inside each case (no dynamic register indexing).
//
// Grid-wide sums (if-else-add's predicate) end a section with a bounded grid barrier in
// a cooperative launch; the branch is then taken on the device (JLE0), no host
// round-trip.
#pragma once
#include <cuda_runtime.h>

#include "dvm_internal.h"
#include "vm_common.cuh"

namespace dvm {

constexpr int NW = kVmWarps;           // consumer warps
constexpr int NTHREADS = (NW + 1) * 32;
constexpr int REG = kVmReg;            // fp32 values per slot per thread
constexpr int kImageSmem = kMaxImage;  // bytes reserved for the image copy
constexpr int kBarOff = kImageSmem;    // 17 mbarriers (8 full, 8 empty, 1 hoist)
constexpr int kRedOff = kBarOff + 256;
constexpr int kRowOff = kRedOff + 256;
constexpr int kMiscOff = kRowOff + 256;
constexpr int kDataOff = kMiscOff + 256;  // hoist area, then the stage ring

struct LaunchParams {
  alignas(16) uint8_t image[kMaxImage];
  void* ptrs[kMaxBind];
  unsigned long long* barrier;
  int32_t* status;
  float* partials;
  unsigned long long barrier_target;
  unsigned long long timeout_ns;
  int32_t skip_arrival;
};

// -------------------------------------------------------------------------
struct Prog {
  const ProgRec* pr;
  const TensRec* tens;
  const Instr* body;   // first instruction of the program body (TILES ...)
  int r, t_in, m, segs, rows;
  int tiles[4];
};

__device__ __forceinline__ void load_prog(const uint8_t* img, int p, Prog& P, int a) {
  P.pr = reinterpret_cast<const ProgRec*>(img + sizeof(Header) + p * sizeof(ProgRec));
  P.tens = reinterpret_cast<const TensRec*>(img + P.pr->tens_off);
  P.body = reinterpret_cast<const Instr*>(img + P.pr->body_off);
  P.r = P.pr->rank;
  P.t_in = (int)P.pr->t[P.r - 1];
  P.m = P.t_in / a;
  P.rows = 1;
  for (int d = 0; d < P.r - 1; d++) P.rows *= (int)P.pr->t[d];
  P.segs = P.rows * P.m;
  for (int d = 0; d < 4; d++) P.tiles[d] = (int)((P.pr->n[d] + P.pr->t[d] - 1) / P.pr->t[d]);
}

// tile origin for local tile index tau (row-major over the tile grid)
__device__ __forceinline__ void tile_origin(const Prog& P, int tau, int o[4]) {
  for (int d = P.r - 1; d >= 0; d--) {
    int td = P.tiles[d];
    int cd = tau % td;
    tau /= td;
    o[d] = cd * (int)P.pr->t[d];
  }
  for (int d = P.r; d < 4; d++) o[d] = 0;
}

// does a section body contain a stage (DMA, non-hoisted) load?
__device__ __forceinline__ bool section_has_stage(const Instr* b, int n) {
  for (int i = 0; i < n; i++)
    if (b[i].op == OP_LD && (b[i].flags & LF_DMA) && !(b[i].flags & LF_HOIST)) return true;
  return false;
}

// element offset of tile row `row` (outer coordinates) for tensor view vs; returns
// false when the row lies outside the iteration space
__device__ __forceinline__ bool row_offset(const Prog& P, const int o[4], int row, const int64_t* vs, int64_t& off) {
  off = 0;
  int rr = row;
  for (int d = P.r - 2; d >= 0; d--) {
    int td = (int)P.pr->t[d];
    int i = o[d] + rr % td;
    rr /= td;
    if (i >= (int)P.pr->n[d]) return false;
    off += (int64_t)i * vs[d];
  }
  return true;
}

// ============================================================== producer ==
// Bulk copies of one tile's DMA loads (or of the hoisted loads when hoist_pass).
// mode 0 counts the bytes, mode 1 issues the copies; the caller arms the mbarrier with
// the counted total in between.
static __device__ uint32_t produce_tile(const LaunchParams& Pm, const Prog& P, const Instr* body, int n, int tau,
                                 uint8_t* dst_base, uint64_t* bar, bool hoist_pass, int mode) {
  int o[4];
  if (hoist_pass) {
    for (int d = 0; d < 4; d++) o[d] = 0;
  } else {
    tile_origin(P, tau, o);
  }
  const int r = P.r;
  const int n_in = (int)P.pr->n[r - 1];
  const int o_in = o[r - 1];
  const int valid_in = min(P.t_in, n_in - o_in);
  uint32_t total = 0;
  for (int i = 0; i < n; i++) {
    const Instr w = body[i];
    if (w.op != OP_LD || !(w.flags & LF_DMA) || !(w.flags & LF_FIRST)) continue;
    if (((w.flags & LF_HOIST) != 0) != hoist_pass) continue;
    const TensRec& T = P.tens[w.b];
    const int esz = dtype_size(T.dtype);
    const uint32_t bytes = (uint32_t)valid_in * esz;
    const int nrows = (w.flags & LF_COLV) ? 1 : P.rows;
    const uint8_t* src = static_cast<const uint8_t*>(Pm.ptrs[T.binding]);
    uint8_t* dst = dst_base + w.aux0;
    for (int row = 0; row < nrows; row++) {
      int64_t off;
      if (!row_offset(P, o, row, T.vs, off)) continue;
      total += bytes;
      if (mode == 1) {
        off += (int64_t)o_in;  // inner stride is 1 for DMA loads
        bulk_g2s(dst + (size_t)row * P.t_in * esz, src + off * esz, bytes, bar);
      }
    }
  }
  return total;
}

// ============================================================== consumer ==
template <int VE>
struct Lanes {
  static constexpr int NV = REG / VE;  // vectors (segments) per thread per slot
  int row[NV];    // tile row of each vector
  int col[NV];    // first tile column of this lane's VE elements
  bool seg[NV];   // vector maps to a segment of the tile
  // per tile
  bool rowok[NV];
  int ncol[NV];   // valid elements among the VE
};

template <int VE>
__device__ __forceinline__ void lanes_for_prog(const Prog& P, int warp, int lane, Lanes<VE>& L) {
  const int a = VE * 32;
#pragma unroll
  for (int v = 0; v < Lanes<VE>::NV; v++) {
    int s = v * NW + warp;
    L.seg[v] = s < P.segs;
    L.row[v] = s / P.m;
    L.col[v] = (s % P.m) * a + lane * VE;
  }
}

template <int VE>
__device__ __forceinline__ void lanes_for_tile(const Prog& P, const int o[4], Lanes<VE>& L) {
  const int r = P.r;
  const int n_in = (int)P.pr->n[r - 1];
#pragma unroll
  for (int v = 0; v < Lanes<VE>::NV; v++) {
    bool ok = L.seg[v];
    int rr = L.row[v];
    for (int d = r - 2; d >= 0 && ok; d--) {
      int td = (int)P.pr->t[d];
      if (o[d] + rr % td >= (int)P.pr->n[d]) ok = false;
      rr /= td;
    }
    L.rowok[v] = ok;
    int nc = n_in - (o[r - 1] + L.col[v]);
    L.ncol[v] = nc < 0 ? 0 : (nc > VE ? VE : nc);
  }
}

// ---- loads into a register slot -------------------------------------------
template <int VE, int ESZ>
__device__ __forceinline__ void unpack(const uint8_t* p, float* dst) {
  // p is 16-byte aligned, VE*ESZ bytes
  if constexpr (ESZ == 4) {
#pragma unroll
    for (int q = 0; q < VE / 4; q++) {
      float4 f = reinterpret_cast<const float4*>(p)[q];
      dst[4 * q] = f.x; dst[4 * q + 1] = f.y; dst[4 * q + 2] = f.z; dst[4 * q + 3] = f.w;
    }
  } else if constexpr (ESZ == 2) {
#pragma unroll
    for (int q = 0; q < VE / 8; q++) {
      uint4 u = reinterpret_cast<const uint4*>(p)[q];
      dst[8 * q + 0] = bf16lo(u.x); dst[8 * q + 1] = bf16hi(u.x);
      dst[8 * q + 2] = bf16lo(u.y); dst[8 * q + 3] = bf16hi(u.y);
      dst[8 * q + 4] = bf16lo(u.z); dst[8 * q + 5] = bf16hi(u.z);
      dst[8 * q + 6] = bf16lo(u.w); dst[8 * q + 7] = bf16hi(u.w);
    }
  } else {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < VE; e++) dst[e] = (float)((w4[e / 4] >> (8 * (e % 4))) & 0xffu);
  }
}

__device__ __forceinline__ float load_scalar(const uint8_t* base, int64_t off, int dt) {
  if (dt == DT_F32) return __ldg(reinterpret_cast<const float*>(base) + off);
  if (dt == DT_BF16) return __uint_as_float(((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(base) + off)) << 16);
  return (float)__ldg(base + off);
}

template <int VE>
__device__ __forceinline__ void op_load(float (&dst)[REG], const Instr& w, const Prog& P, const Lanes<VE>& L,
                                        const int o[4], const LaunchParams& Pm, const uint8_t* stage_base,
                                        const uint8_t* hoist_base) {
  const TensRec& T = P.tens[w.b];
  const int dt = T.dtype;
  const int esz = dtype_size(dt);
  if (w.flags & LF_DMA) {
    const uint8_t* region = ((w.flags & LF_HOIST) ? hoist_base + P.pr->hoist_base : stage_base) + w.aux0;
    const bool colv = (w.flags & LF_COLV) != 0;
#pragma unroll
    for (int v = 0; v < Lanes<VE>::NV; v++) {
      if (!L.seg[v]) continue;
      const uint8_t* p = region + ((colv ? 0 : (size_t)L.row[v] * P.t_in) + L.col[v]) * esz;
      if (esz == 4) unpack<VE, 4>(p, dst + v * VE);
      else if (esz == 2) {
        if constexpr (VE >= 8) unpack<VE, 2>(p, dst + v * VE);
      } else {
        if constexpr (VE == 16) unpack<VE, 1>(p, dst + v * VE);
      }
    }
    return;
  }
  // direct loads from global memory
  const uint8_t* base = static_cast<const uint8_t*>(Pm.ptrs[T.binding]);
  const int r = P.r;
  const int64_t vin = T.vs[r - 1];
  const bool rowv = (w.flags & LF_ROWV) != 0;
#pragma unroll
  for (int v = 0; v < Lanes<VE>::NV; v++) {
    float* d = dst + v * VE;
    int64_t off;
    if (!L.seg[v] || !L.rowok[v] || !row_offset(P, o, L.row[v], T.vs, off)) {
#pragma unroll
      for (int e = 0; e < VE; e++) d[e] = 0.f;
      continue;
    }
    if (rowv) {
      d[0] = load_scalar(base, off, dt);
      continue;
    }
    off += (int64_t)(o[r - 1] + L.col[v]) * vin;
    if (vin == 1 && L.ncol[v] == VE && ((off * esz) & 15) == 0) {
      const uint8_t* p = base + off * esz;
      if (esz == 4) unpack<VE, 4>(p, d);
      else if (esz == 2) {
        if constexpr (VE >= 8) unpack<VE, 2>(p, d);
      } else {
        if constexpr (VE == 16) unpack<VE, 1>(p, d);
      }
    } else {
#pragma unroll
      for (int e = 0; e < VE; e++) d[e] = e < L.ncol[v] ? load_scalar(base, off + e * vin, dt) : 0.f;
    }
  }
}

// ---- stores from ACC --------------------------------------------------------
__device__ __forceinline__ void store_scalar(uint8_t* base, int64_t off, int dt, float x) {
  if (dt == DT_F32) reinterpret_cast<float*>(base)[off] = x;
  else if (dt == DT_BF16) reinterpret_cast<__nv_bfloat16*>(base)[off] = __float2bfloat16_rn(x);
  else base[off] = (uint8_t)(x != 0.f ? 1 : 0);
}

template <int VE>
__device__ __forceinline__ void op_store(const float (&acc)[REG], const Instr& w, const Prog& P, const Lanes<VE>& L,
                                         const int o[4], const LaunchParams& Pm) {
  const TensRec& T = P.tens[w.a];
  const int dt = T.dtype;
  const int esz = dtype_size(dt);
  uint8_t* base = static_cast<uint8_t*>(Pm.ptrs[T.binding]);
  const int r = P.r;
  const int64_t vin = T.vs[r - 1];
  const bool rowv = (w.flags & LF_ROWV) != 0;
#pragma unroll
  for (int v = 0; v < Lanes<VE>::NV; v++) {
    int64_t off;
    if (!L.seg[v] || !L.rowok[v]) continue;
    if (rowv && L.col[v] != 0) continue;  // one writer per row
    if (!row_offset(P, o, L.row[v], T.vs, off)) continue;
    const float* s = acc + v * VE;
    if (rowv) {
      store_scalar(base, off, dt, s[0]);
      continue;
    }
    off += (int64_t)(o[r - 1] + L.col[v]) * vin;
    if (vin == 1 && L.ncol[v] == VE && ((off * esz) & 15) == 0) {
      uint8_t* p = base + off * esz;
      if (esz == 4) {
#pragma unroll
        for (int q = 0; q < VE / 4; q++)
          reinterpret_cast<float4*>(p)[q] = make_float4(s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3]);
      } else if (esz == 2) {
        if constexpr (VE >= 8) {
#pragma unroll
          for (int q = 0; q < VE / 8; q++) {
            uint4 u;
            u.x = pack_bf16(s[8 * q], s[8 * q + 1]);
            u.y = pack_bf16(s[8 * q + 2], s[8 * q + 3]);
            u.z = pack_bf16(s[8 * q + 4], s[8 * q + 5]);
            u.w = pack_bf16(s[8 * q + 6], s[8 * q + 7]);
            reinterpret_cast<uint4*>(p)[q] = u;
          }
        }
      } else {
        if constexpr (VE == 16) {
          uint32_t w4[4] = {0, 0, 0, 0};
#pragma unroll
          for (int e = 0; e < 16; e++) w4[e / 4] |= (uint32_t)(s[e] != 0.f ? 1 : 0) << (8 * (e % 4));
          *reinterpret_cast<uint4*>(p) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < VE; e++)
        if (e < L.ncol[v]) store_scalar(base, off + e * vin, dt, s[e]);
    }
  }
}

// ---- element-wise math --------------------------------------------------------
__device__ __forceinline__ float unary_fn(int op, float x) {
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
    case OP_CASTBF: return round_bf16(x);
    default: return x;
  }
}
// out-of-line scalar paths keep rarely used or large code out of the unrolled loops
static __device__ __noinline__ float unary_scalar(int op, float x) { return unary_fn(op, x); }
static __device__ __noinline__ float pow_scalar(float a, float b) { return powf(a, b); }

template <int OP>
__device__ __forceinline__ float bin(float a, float b) {
  if constexpr (OP == OP_ADD) return a + b;
  else if constexpr (OP == OP_SUB) return a - b;
  else if constexpr (OP == OP_MUL) return a * b;
  else if constexpr (OP == OP_DIV) return a / b;
  else if constexpr (OP == OP_MAX) return vmax(a, b);
  else if constexpr (OP == OP_MIN) return vmin(a, b);
  else return pow_scalar(a, b);
}

template <int OP>
__device__ __forceinline__ float bin_r(float a, float x, bool rev) {
  if constexpr (OP == OP_ADD || OP == OP_MUL || OP == OP_MAX || OP == OP_MIN) return bin<OP>(a, x);
  else return rev ? bin<OP>(x, a) : bin<OP>(a, x);
}

// ACC <- op(ACC, X) with row/full kinds; X is a slot
template <int VE, int OP>
__device__ __forceinline__ void bin_slot(float (&acc)[REG], const float (&x)[REG], uint8_t fl) {
  constexpr int NV = REG / VE;
  const bool rev = fl & CF_REV;
  const bool ar = fl & CF_AROW, xr = fl & CF_XROW;
  if (ar && xr) {
#pragma unroll
    for (int v = 0; v < NV; v++) acc[v * VE] = bin_r<OP>(acc[v * VE], x[v * VE], rev);
  } else if (ar) {
#pragma unroll
    for (int v = 0; v < NV; v++) {
      float a0 = acc[v * VE];
#pragma unroll
      for (int e = 0; e < VE; e++) acc[v * VE + e] = bin_r<OP>(a0, x[v * VE + e], rev);
    }
  } else if (xr) {
#pragma unroll
    for (int v = 0; v < NV; v++) {
      float x0 = x[v * VE];
#pragma unroll
      for (int e = 0; e < VE; e++) acc[v * VE + e] = bin_r<OP>(acc[v * VE + e], x0, rev);
    }
  } else {
#pragma unroll
    for (int e = 0; e < REG; e++) acc[e] = bin_r<OP>(acc[e], x[e], rev);
  }
}

template <int VE, int OP>
__device__ __forceinline__ void bin_imm(float (&acc)[REG], float x, uint8_t fl) {
  constexpr int NV = REG / VE;
  const bool rev = fl & CF_REV;
  if (fl & CF_AROW) {
#pragma unroll
    for (int v = 0; v < NV; v++) acc[v * VE] = bin_r<OP>(acc[v * VE], x, rev);
  } else {
#pragma unroll
    for (int e = 0; e < REG; e++) acc[e] = bin_r<OP>(acc[e], x, rev);
  }
}

template <int VE, int OP>
__device__ __forceinline__ void do_bin(float (&R0)[REG], float (&R1)[REG], float (&R2)[REG], const Instr& w) {
  if (w.flags & CF_IMM) {
    bin_imm<VE, OP>(R0, __uint_as_float(w.imm), w.flags);
    return;
  }
  switch (w.a) {
    case 0: bin_slot<VE, OP>(R0, R0, w.flags); break;
    case 1: bin_slot<VE, OP>(R0, R1, w.flags); break;
    default: bin_slot<VE, OP>(R0, R2, w.flags); break;
  }
}

__device__ __forceinline__ void copy_slot(float (&d)[REG], const float (&s)[REG]) {
#pragma unroll
  for (int e = 0; e < REG; e++) d[e] = s[e];
}

// warp-level all-reduce (xor butterfly: every lane ends with identical bits)
template <bool MAX>
__device__ __forceinline__ float warp_reduce(float p) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float q = __shfl_xor_sync(0xffffffffu, p, o);
    p = MAX ? vmax(p, q) : p + q;
  }
  return p;
}

// ACC (FULL) -> ACC (ROW): reduce each tile row over its valid columns.
// Order is fixed: each lane sums its VE elements in order, the warp butterfly combines
// the 32 lanes of a segment, then the segments of a row are combined by one warp.
template <int VE, bool MAX>
__device__ __forceinline__ void row_reduce(float (&acc)[REG], const Prog& P, const Lanes<VE>& L, int warp, int lane,
                                           float* red, float* rowtot) {
  constexpr int NV = REG / VE;
  const float ident = MAX ? -INFINITY : 0.f;
#pragma unroll
  for (int v = 0; v < NV; v++) {
    float p = ident;
    if (L.seg[v] && L.rowok[v]) {
#pragma unroll
      for (int e = 0; e < VE; e++)
        if (e < L.ncol[v]) p = MAX ? vmax(p, acc[v * VE + e]) : p + acc[v * VE + e];
    }
    p = warp_reduce<MAX>(p);
    if (lane == 0 && L.seg[v]) red[v * NW + warp] = p;
  }
  named_bar(1, NW * 32);
  for (int row = warp; row < P.rows; row += NW) {
    float q = ident;
    for (int j = lane; j < P.m; j += 32) q = MAX ? vmax(q, red[row * P.m + j]) : q + red[row * P.m + j];
    q = warp_reduce<MAX>(q);
    if (lane == 0) rowtot[row] = q;
  }
  named_bar(1, NW * 32);
#pragma unroll
  for (int v = 0; v < NV; v++)
    if (L.seg[v]) acc[v * VE] = rowtot[L.row[v]];
}

// ---- one tile -------------------------------------------------------------
struct Ctl {
  uint64_t* full;
  uint64_t* empty;
  int n_stages;
  uint32_t stage_bytes;
  uint8_t* ring;
  uint8_t* hoist;
  volatile int* abort;
  DevStatus st;
};

template <int VE>
__device__ __forceinline__ void exec_tile(const LaunchParams& Pm, const Prog& P, const Instr* body, int n, int tau,
                                          Lanes<VE>& L, int warp, int lane, int it, const Ctl& C, float* red,
                                          float* rowtot, float& grand, float (&R0)[REG], float (&R1)[REG],
                                          float (&R2)[REG]) {
  constexpr int NV = REG / VE;
  int o[4];
  tile_origin(P, tau, o);
  lanes_for_tile<VE>(P, o, L);
  const int stage = C.n_stages ? it % C.n_stages : 0;
  const uint32_t parity = C.n_stages ? (uint32_t)((it / C.n_stages) & 1) : 0;
  const uint8_t* stage_base = C.ring + (size_t)stage * C.stage_bytes;
  for (int pc = 0; pc < n; pc++) {
    const Instr w = body[pc];
    switch (w.op) {
      case OP_WAIT:
        mbar_wait(&C.full[stage], parity, C.st, C.abort);
        break;
      case OP_REL:
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.empty[stage]);
        break;
      case OP_LD:
        switch (w.a) {
          case 0: op_load<VE>(R0, w, P, L, o, Pm, stage_base, C.hoist); break;
          case 1: op_load<VE>(R1, w, P, L, o, Pm, stage_base, C.hoist); break;
          default: op_load<VE>(R2, w, P, L, o, Pm, stage_base, C.hoist); break;
        }
        break;
      case OP_ST:
        op_store<VE>(R0, w, P, L, o, Pm);
        break;
      case OP_MOV:
        if (w.a == 0) {
          if (w.b == 1) copy_slot(R0, R1);
          else if (w.b == 2) copy_slot(R0, R2);
        } else if (w.a == 1) {
          copy_slot(R1, R0);
        } else {
          copy_slot(R2, R0);
        }
        break;
      case OP_BCAST:
#pragma unroll
        for (int v = 0; v < NV; v++)
#pragma unroll
          for (int e = 1; e < VE; e++) R0[v * VE + e] = R0[v * VE];
        break;
      case OP_ADD: do_bin<VE, OP_ADD>(R0, R1, R2, w); break;
      case OP_SUB: do_bin<VE, OP_SUB>(R0, R1, R2, w); break;
      case OP_MUL: do_bin<VE, OP_MUL>(R0, R1, R2, w); break;
      case OP_DIV: do_bin<VE, OP_DIV>(R0, R1, R2, w); break;
      case OP_MAX: do_bin<VE, OP_MAX>(R0, R1, R2, w); break;
      case OP_MIN: do_bin<VE, OP_MIN>(R0, R1, R2, w); break;
      case OP_POW: do_bin<VE, OP_POW>(R0, R1, R2, w); break;
      case OP_RSUM: row_reduce<VE, false>(R0, P, L, warp, lane, red, rowtot); break;
      case OP_RMAX: row_reduce<VE, true>(R0, P, L, warp, lane, red, rowtot); break;
      case OP_ASUM:
        if (w.flags & CF_AROW) {
#pragma unroll
          for (int v = 0; v < NV; v++)
            if (L.seg[v] && L.rowok[v] && L.col[v] == 0) grand += R0[v * VE];
        } else {
#pragma unroll
          for (int v = 0; v < NV; v++)
            if (L.seg[v] && L.rowok[v]) {
#pragma unroll
              for (int e = 0; e < VE; e++)
                if (e < L.ncol[v]) grand += R0[v * VE + e];
            }
        }
        break;
      case OP_SQRT: case OP_ABS: case OP_LOG: case OP_EXP: case OP_ROUND: case OP_FLOOR:
      case OP_ISFIN: case OP_NEG: case OP_RSQRT: case OP_RECIP: case OP_SILU: case OP_CASTBF: {
        const int op = w.op;
        if (w.flags & CF_AROW) {
#pragma unroll
          for (int v = 0; v < NV; v++) R0[v * VE] = unary_scalar(op, R0[v * VE]);
        } else {
          switch (op) {  // one loop per opcode keeps the math inlined and branch-free
#define DVM_UNARY_CASE(OPC)                                                        \
  case OPC:                                                                        \
    _Pragma("unroll") for (int e = 0; e < REG; e++) R0[e] = unary_fn(OPC, R0[e]); \
    break;
            DVM_UNARY_CASE(OP_SQRT) DVM_UNARY_CASE(OP_ABS) DVM_UNARY_CASE(OP_LOG) DVM_UNARY_CASE(OP_EXP)
            DVM_UNARY_CASE(OP_ROUND) DVM_UNARY_CASE(OP_FLOOR) DVM_UNARY_CASE(OP_ISFIN) DVM_UNARY_CASE(OP_NEG)
            DVM_UNARY_CASE(OP_RSQRT) DVM_UNARY_CASE(OP_RECIP) DVM_UNARY_CASE(OP_SILU) DVM_UNARY_CASE(OP_CASTBF)
#undef DVM_UNARY_CASE
            default: break;
          }
        }
        break;
      }
      default:
        set_status(Pm.status, -101 /* DVM_E_BAD_OPCODE */);
        break;
    }
  }
}

// ---- grid-wide sum (GSUM) -------------------------------------------------
// Called by every thread of the CTA. Consumers pass their grand sums; the result is
// identical on every CTA (fixed combination order). The wait for the other CTAs is
// bounded; on expiry the status word is set and every thread of the CTA sees `abort`.
static __device__ __noinline__ float grid_sum(const LaunchParams& Pm, float grand, bool consumer, int warp, int lane,
                                       float* red, float* misc_s, volatile int* abort) {
  if (consumer) {
    float p = warp_reduce<false>(grand);
    if (lane == 0) red[warp] = p;
    named_bar(1, NW * 32);
    if (threadIdx.x == 0) {
      float cta = 0.f;
      for (int w = 0; w < NW; w++) cta += red[w];
      Pm.partials[blockIdx.x] = cta;
      __threadfence();
      if (!(Pm.skip_arrival && blockIdx.x == 0)) atomicAdd(Pm.barrier, 1ull);
      unsigned long long t0 = globaltimer();
      while (true) {
        unsigned long long v = *reinterpret_cast<volatile unsigned long long*>(Pm.barrier);
        if (v >= Pm.barrier_target) break;
        if (globaltimer() - t0 > Pm.timeout_ns) {
          set_status(Pm.status, -100 /* DVM_E_TIMEOUT */);
          *abort = 1;
          break;
        }
        __nanosleep(256);
      }
      __threadfence();
    }
  }
  __syncthreads();
  if (*abort) return 0.f;
  if (consumer && warp == 0) {
    float q = 0.f;
    for (int c = lane; c < (int)gridDim.x; c += 32) q += __ldcg(Pm.partials + c);
    q = warp_reduce<false>(q);
    if (lane == 0) *misc_s = q;
  }
  __syncthreads();
  return *misc_s;
}

// Walks the launch's work in order — plain/stacked: the CTA's range of the concatenated
// tile list; sectioned: the top-level control flow (TILES / GSUM / SST / JLE0 / JMP /
// END) — and yields one (program, section, tile) at a time.  Producer and consumers
// run the same walker, so they agree on the stage sequence.
struct Walker {
  const uint8_t* img;
  const Header* H;
  int a, lo, hi;
  bool sectioned, consumer;
  // current position
  Prog P;
  int p = -1;
  int g = 0;            // plain: next concatenated tile
  int pc = 0;           // sectioned: next top-level instruction
  int tau = 0, t_end = 0;
  const Instr* sec = nullptr;
  int sec_n = 0;
  bool stage = false;   // current section has stage loads
  float S = 0.f;

  __device__ __forceinline__ void init(const uint8_t* image, int a_, bool cons) {
    img = image;
    H = reinterpret_cast<const Header*>(image);
    a = a_;
    consumer = cons;
    lo = blockIdx.x * (int)H->body_tile;
    hi = min(lo + (int)H->body_tile, (int)H->block_dim);
    sectioned = reinterpret_cast<const ProgRec*>(image + sizeof(Header))->kind == PK_SEC;
    g = lo;
    if (sectioned) {
      p = 0;
      load_prog(img, 0, P, a);
      tau = t_end = 0;
    }
  }
  // returns false when the CTA's work is done; `changed` = program changed
  template <class OnGsum>
  __device__ __forceinline__ bool next(int& out_tau, bool& changed, OnGsum on_gsum, const LaunchParams& Pm,
                                       volatile int* abort) {
    changed = false;
    if (!sectioned) {
      if (g >= hi) return false;
      if (p < 0 || g >= (int)(P.pr->tile_base + P.pr->block_dim)) {
        for (int q = 0; q < H->n_progs; q++) {
          const ProgRec* pr = reinterpret_cast<const ProgRec*>(img + sizeof(Header) + q * sizeof(ProgRec));
          if (g >= (int)pr->tile_base && g < (int)(pr->tile_base + pr->block_dim)) {
            p = q;
            break;
          }
        }
        load_prog(img, p, P, a);
        sec = P.body + 1;
        sec_n = (int)P.body[0].imm;
        stage = section_has_stage(sec, sec_n);
        changed = true;
      }
      out_tau = g - (int)P.pr->tile_base;
      g++;
      return true;
    }
    while (tau >= t_end) {
      if (pc >= (int)P.pr->body_len) return false;
      const Instr w = P.body[pc];
      if (w.op == OP_TILES) {
        sec = P.body + pc + 1;
        sec_n = (int)w.imm;
        stage = section_has_stage(sec, sec_n);
        tau = lo;
        t_end = min(hi, (int)P.pr->block_dim);
        pc += 1 + sec_n;
        changed = true;
      } else if (w.op == OP_GSUM) {
        S = on_gsum();
        if (*abort) return false;
        pc++;
      } else if (w.op == OP_SST) {
        if (consumer && blockIdx.x == 0 && threadIdx.x == 0) {
          const TensRec& T = P.tens[w.a];
          store_scalar(static_cast<uint8_t*>(Pm.ptrs[T.binding]), 0, T.dtype, S);
        }
        pc++;
      } else if (w.op == OP_JLE0) {
        pc += 1 + (S > 0.f ? 0 : (int)w.imm);
      } else if (w.op == OP_JMP) {
        pc += 1 + (int)w.imm;
      } else {
        return false;  // END
      }
    }
    out_tau = tau++;
    return true;
  }
};

// ---- the kernel --------------------------------------------------------------
template <int VE>
__global__ void __launch_bounds__(NTHREADS, 1) vm_vec_kernel(const __grid_constant__ LaunchParams Pm) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  {
    const uint32_t total = reinterpret_cast<const Header*>(Pm.image)->total_len;
    for (uint32_t i = tid * 16; i < total; i += NTHREADS * 16)
      *reinterpret_cast<uint4*>(smem + i) = *reinterpret_cast<const uint4*>(Pm.image + i);
  }
  const Header* H = reinterpret_cast<const Header*>(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* full = bars;
  uint64_t* empty = bars + 8;
  uint64_t* hbar = bars + 16;
  float* red = reinterpret_cast<float*>(smem + kRedOff);
  float* rowtot = reinterpret_cast<float*>(smem + kRowOff);
  float* misc_s = reinterpret_cast<float*>(smem + kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kMiscOff + 16);
  if (tid == 0) {
    for (int s = 0; s < 8; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    mbar_init(hbar, 1);
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  Ctl C;
  C.full = full;
  C.empty = empty;
  C.n_stages = H->n_stages;
  C.stage_bytes = H->stage_bytes;
  C.hoist = smem + kDataOff;
  C.ring = smem + kDataOff + ((H->hoist_bytes + 127) & ~127u);
  C.abort = abort;
  C.st.word = Pm.status;
  C.st.limit_ns = Pm.timeout_ns;

  const int a = VE * 32;
  const bool producer = warp == NW;
  Walker W;
  W.init(smem, a, !producer);
  const bool has_work = W.lo < W.hi;

  if (producer) {
    // ----------------------------------------------------------- DMA flow
    const bool leader = lane == 0;
    if (leader && H->hoist_bytes && has_work) {
      // hoisted (tile-invariant) loads: once per CTA, all programs, one mbarrier phase
      uint32_t total = 0;
      for (int mode = 0; mode < 2; mode++) {
        if (mode == 1) mbar_arrive_expect_tx(hbar, total);
        for (int p = 0; p < H->n_progs; p++) {
          Prog P;
          load_prog(smem, p, P, a);
          total += produce_tile(Pm, P, P.body, (int)P.pr->body_len, 0, C.hoist + P.pr->hoist_base, hbar, true, mode);
        }
      }
    } else if (leader) {
      mbar_arrive(hbar);
    }
    int it = 0;
    int tau;
    bool changed;
    auto gsum = [&]() { return grid_sum(Pm, 0.f, false, warp, lane, red, misc_s, abort); };
    while (W.next(tau, changed, gsum, Pm, abort)) {
      if (!W.stage) continue;
      const int stage = it % C.n_stages;
      const uint32_t parity = ((it / C.n_stages) & 1) ^ 1;
      if (leader && !*abort && mbar_wait(&empty[stage], parity, C.st, abort)) {
        uint8_t* dst = C.ring + (size_t)stage * C.stage_bytes;
        const uint32_t bytes = produce_tile(Pm, W.P, W.sec, W.sec_n, tau, dst, &full[stage], false, 0);
        mbar_arrive_expect_tx(&full[stage], bytes);
        produce_tile(Pm, W.P, W.sec, W.sec_n, tau, dst, &full[stage], false, 1);
      }
      it++;
    }
    // on an abort, let copies already in flight land before the CTA exits (bounded)
    if (leader && *abort) {
      for (int k = 1; k <= C.n_stages && k <= it; k++) {
        const int s = (it - k) % C.n_stages;
        unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(&full[s], (uint32_t)(((it - k) / C.n_stages) & 1)) && globaltimer() - t0 < 1000000ull) {
        }
      }
    }
    return;
  }

  // --------------------------------------------------------------- vector flow
  float R0[REG], R1[REG], R2[REG];
#pragma unroll
  for (int e = 0; e < REG; e++) { R0[e] = R1[e] = R2[e] = 0.f; }
  float grand = 0.f;
  if (H->hoist_bytes && has_work) mbar_wait(hbar, 0, C.st, abort);
  int it = 0;
  Lanes<VE> L;
  int tau;
  bool changed;
  auto gsum = [&]() { return grid_sum(Pm, grand, true, warp, lane, red, misc_s, abort); };
  while (W.next(tau, changed, gsum, Pm, abort)) {
    if (changed) lanes_for_prog<VE>(W.P, warp, lane, L);
    exec_tile<VE>(Pm, W.P, W.sec, W.sec_n, tau, L, warp, lane, it, C, red, rowtot, grand, R0, R1, R2);
    if (W.stage) it++;
  }
}

// host-side launcher for one lane width (instantiated in vm_vec<VE>.cu)
template <int VE>
cudaError_t launch_vec(const LaunchParams& P, int grid, size_t smem, bool coop, cudaStream_t s) {
  static bool attr_done = false;
  auto k = vm_vec_kernel<VE>;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  if (coop) {
    void* args[] = {const_cast<LaunchParams*>(&P)};
    return cudaLaunchCooperativeKernel((const void*)k, dim3(grid), dim3(NTHREADS), args, smem, s);
  }
  k<<<grid, NTHREADS, smem, s>>>(P);
  return cudaGetLastError();
}

}  // namespace dvm
