// vm_vec.cuh — the persistent DVM interpreter for element-wise / reduce programs (VEC
// kernel type), sm_103a.
//
// Execution model (DVM review page, section 4.4 "virtual machine execution"): each CTA
// is one "AI core"; it computes its contiguous tile range [c*body_tile,
// min((c+1)*body_tile, block_dim)) and, for each tile, decodes the code body and calls
// the matching virtual-instruction function.  Decoding is warp-uniform from the image
// staged in shared memory.  Section 3.2's asynchronous flows map onto one CTA:
//   * DMA flow    -> thread 0 keeps a ring of shared-memory stages filled S-1 tiles
//                    ahead with cp.async.bulk copies, signalled by mbarriers;
//   * vector flow -> 8 warps move a tile from its stage into registers (LD), run the
//                    element-wise chain in registers, reduce rows with warp shuffles,
//                    and store from registers straight to HBM (ST);
//   * the WAIT / REL words the encoder inserts are the syncs between the two flows.
//
// Registers follow an accumulator machine: ACC (REG = 32 fp32 values per thread in
// registers) plus 2 addressable slots held in per-thread shared-memory storage.  Every
// instruction reads ACC and at most one slot, so no register is ever indexed at run time.
// Values of ROW kind (one per tile row: row sums, means, rstd) do not live in
// registers: they live in three shared-memory row buffers (ACC, slot 1, slot 2) and
// are computed once per row by one thread, then read by the element-wise ops.
//
// Grid-wide sums (if-else-add's predicate) end a section with a bounded grid barrier in
// a cooperative launch; the branch is then taken on the device (JLE0), no host
// round-trip.
#pragma once
#include <cuda_runtime.h>

#include "dvm_internal.h"
#include "vm_common.cuh"

namespace dvm {

constexpr int NW = kVmWarps;          // warps per CTA
constexpr int NTHREADS = NW * 32;
constexpr int REG = kVmReg;           // fp32 values per slot per thread
constexpr int kMaxRows = 64;          // rows per tile (a >= 128 elements, cap 8192)
// shared memory layout
constexpr int kBarOff = kMaxImage;                    // 17 mbarriers (8 full, 8 empty, 1 hoist)
constexpr int kRedOff = kBarOff + 256;                // per (row, warp) partial sums
constexpr int kRowBufOff = kRedOff + kMaxRows * NW * 4;  // 3 row buffers: ACC, slot 1, slot 2
constexpr int kRowCoordOff = kRowBufOff + 3 * kMaxRows * 4;  // outer coordinates of each tile row
constexpr int kIssOff = kRowCoordOff + kMaxRows * 4 * 4;  // producer state
constexpr int kMiscOff = kIssOff + 256;
constexpr int kSlotOff = kMiscOff + 128;              // slots 1, 2 and a scratch slot 3 (per thread)
constexpr int kDataOff = kSlotOff + 3 * REG * 4 * NTHREADS;  // hoist area, then the stage ring
static_assert(kDataOff % 128 == 0, "data area alignment");
static_assert(kDataOff + kSmemBudget <= 227 * 1024, "shared memory of the VEC interpreter");

// the CTA's dynamic shared memory (image copy, barriers, reduction scratch, data)
extern __shared__ __align__(1024) uint8_t dvm_smem[];

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

// ------------------------------------------------------------------ program --
struct Prog {
  const ProgRec* pr;
  const TensRec* tens;
  const Instr* body;   // TILES at body[0] for plain programs
  int r, t_in, m, segs, rows;
  int n0, t0, n_in, tiles_in;  // rank <= 2 fast path: outer extent/tile, inner extent, inner tiles
};

__device__ __forceinline__ void load_prog(const uint8_t* img, int p, Prog& P, int a) {
  P.pr = reinterpret_cast<const ProgRec*>(img + sizeof(Header) + p * sizeof(ProgRec));
  P.tens = reinterpret_cast<const TensRec*>(img + P.pr->tens_off);
  P.body = reinterpret_cast<const Instr*>(img + P.pr->body_off);
  P.r = P.pr->rank;
  P.t_in = (int)P.pr->t[P.r - 1];
  P.n_in = (int)P.pr->n[P.r - 1];
  P.m = P.t_in / a;
  P.rows = 1;
  for (int d = 0; d < P.r - 1; d++) P.rows *= (int)P.pr->t[d];
  P.segs = P.rows * P.m;
  P.tiles_in = (P.n_in + P.t_in - 1) / P.t_in;
  P.n0 = P.r >= 2 ? (int)P.pr->n[0] : 1;
  P.t0 = P.r >= 2 ? (int)P.pr->t[0] : 1;
}

// Position of a tile: local index tau, its tile coordinates and origin.  Rank <= 2
// tiles are walked incrementally (no division per tile).  Origins are named scalars or
// arrays indexed only by compile-time constants, so nothing lands in local memory.
struct TilePos {
  int tau;
  int c0, cin;   // tile coordinates (rank <= 2)
  int od[3];     // origin of the outer dims 0..2 (dims >= rank-1 unused)
  int oin;       // origin of the inner dim
};

__device__ __forceinline__ void pos_origin(const Prog& P, TilePos& T) {
  if (P.r <= 2) {
    T.od[0] = P.r == 2 ? T.c0 * P.t0 : 0;
    T.oin = T.cin * P.t_in;
  } else {
    int tau = T.tau;
    T.oin = (tau % P.tiles_in) * P.t_in;
    tau /= P.tiles_in;
#pragma unroll
    for (int dd = 2; dd >= 0; dd--) {
      if (dd < P.r - 1) {
        const int td = (int)((P.pr->n[dd] + P.pr->t[dd] - 1) / P.pr->t[dd]);
        T.od[dd] = (tau % td) * (int)P.pr->t[dd];
        tau /= td;
      }
    }
  }
}
__device__ __forceinline__ void pos_start(const Prog& P, TilePos& T, int tau) {
  T.tau = tau;
  T.c0 = tau / P.tiles_in;
  T.cin = tau - T.c0 * P.tiles_in;
  pos_origin(P, T);
}
__device__ __forceinline__ void pos_next(const Prog& P, TilePos& T) {
  T.tau++;
  if (++T.cin == P.tiles_in) {
    T.cin = 0;
    T.c0++;
  }
  pos_origin(P, T);
}

// outer coordinates (within the tile) of tile row `row`, for rank > 2 programs; filled
// by fill_rowcoords whenever the CTA switches program
__device__ __forceinline__ const int* rowcoord(int row) {
  return reinterpret_cast<const int*>(dvm_smem + kRowCoordOff) + (row & (kMaxRows - 1)) * 4;
}

// element offset of tile row `row` for a tensor view; false if the row is outside
__device__ __forceinline__ bool row_off(const Prog& P, const TilePos& O, int row, const int64_t* vs, int64_t& off) {
  if (P.r == 1) {
    off = 0;
    return true;
  }
  if (P.r == 2) {
    const int i = O.od[0] + row;
    off = (int64_t)i * vs[0];
    return i < P.n0;
  }
  const int* rc = rowcoord(row);
  off = 0;
  bool ok = true;
#pragma unroll
  for (int dd = 0; dd < 3; dd++) {
    if (dd < P.r - 1) {
      const int i = O.od[dd] + rc[dd];
      ok = ok && i < (int)P.pr->n[dd];
      off += (int64_t)i * vs[dd];
    }
  }
  return ok;
}

// the same with divisions and no table, for a tile origin given as scalars (used by the
// producer thread, which may run ahead into another program, and by the hoist pass)
static __device__ __noinline__ bool row_off_div(const ProgRec* pr, int rank, int od0, int od1, int od2, int row,
                                         const int64_t* vs, int64_t* off) {
  int64_t o = 0;
  bool ok = true;
  int rr = row;
  for (int d = rank - 2; d >= 0; d--) {
    const int td = (int)pr->t[d];
    const int i = (d == 0 ? od0 : d == 1 ? od1 : od2) + rr % td;
    rr /= td;
    ok = ok && i < (int)pr->n[d];
    o += (int64_t)i * vs[d];
  }
  *off = o;
  return ok;
}
__device__ __forceinline__ bool row_off_any(const Prog& P, const TilePos& O, int row, const int64_t* vs,
                                            int64_t& off) {
  if (P.r <= 2) return row_off(P, O, row, vs, off);
  return row_off_div(P.pr, P.r, O.od[0], O.od[1], O.od[2], row, vs, &off);
}

// does a section body contain a stage (DMA, non-hoisted) load?
__device__ __forceinline__ bool section_has_stage(const Instr* b, int n) {
  for (int i = 0; i < n; i++)
    if (b[i].op == OP_LD && (b[i].flags & LF_DMA) && !(b[i].flags & LF_HOIST)) return true;
  return false;
}

// =========================================================== DMA flow ==
// Bulk copies of the DMA loads of one tile (or, with hoist_pass, of the hoisted
// loads at origin 0).  mode 0 counts bytes, mode 1 issues; the caller arms the
// mbarrier with the count in between.
__device__ __forceinline__ uint32_t dma_tile(const LaunchParams& Pm, const Prog& P, const Instr* body, int n,
                                             const TilePos& O, uint8_t* dst_base, uint64_t* bar, bool hoist_pass,
                                             int mode) {
  const int r = P.r;
  const int o_in = O.oin;
  const int valid_in = min(P.t_in, P.n_in - o_in);
  uint32_t total = 0;
  for (int i = 0; i < n; i++) {
    const Instr w = body[i];
    if (w.op != OP_LD || (w.flags & (LF_DMA | LF_FIRST)) != (LF_DMA | LF_FIRST)) continue;
    if (((w.flags & LF_HOIST) != 0) != hoist_pass) continue;
    const TensRec& T = P.tens[w.b];
    const int esz = dtype_size(T.dtype);
    const uint8_t* src = static_cast<const uint8_t*>(Pm.ptrs[T.binding]);
    uint8_t* dst = dst_base + w.aux0;
    if (w.flags & LF_COLV) {
      int64_t off;
      if (row_off_any(P, O, 0, T.vs, off)) {
        total += (uint32_t)(valid_in * esz);
        if (mode) bulk_g2s(dst, src + (off + o_in) * esz, (uint32_t)(valid_in * esz), bar);
      }
    } else if (r == 2 && valid_in == P.t_in && T.vs[0] == (int64_t)P.t_in) {
      // whole rows of a row-major tensor: the tile is one contiguous block
      const int nrows = min(P.rows, P.n0 - O.od[0]);
      const uint32_t bytes = (uint32_t)nrows * P.t_in * esz;
      total += bytes;
      if (mode) bulk_g2s(dst, src + ((int64_t)O.od[0] * T.vs[0] + o_in) * esz, bytes, bar);
    } else {
      const uint32_t bytes = (uint32_t)(valid_in * esz);
      for (int row = 0; row < P.rows; row++) {
        int64_t off;
        if (!row_off_any(P, O, row, T.vs, off)) continue;
        total += bytes;
        if (mode) bulk_g2s(dst + (size_t)row * P.t_in * esz, src + (off + o_in) * esz, bytes, bar);
      }
    }
  }
  return total;
}

// Producer state, kept in shared memory (only thread 0 touches it).  The stage loads
// of the current section are described once (source, strides, smem offset, copy shape)
// so that issuing a tile costs a few instructions per copy.
struct DmaEnt {
  const uint8_t* src;  // tensor base
  int64_t vs0;         // outer stride (elements) for rank 2
  uint32_t aux0;       // offset in the stage
  int esz;
  int kind;            // 0 one row (COLV), 1 contiguous block of whole rows, 2 row by row, 3 generic
  int tens;            // program-local tensor index (generic path)
};
struct Issuer {
  int prog;        // program of the next tile to issue (plain mode)
  int g;           // plain: next concatenated tile index
  int g_end;
  int tau, t_end;  // current program-local range
  int c0, cin;
  int sec_off, sec_n;  // section body (instruction index, count)
  int stage_sec;   // the section has stage loads
  int issued;      // staged tiles issued so far
  int n_dma;
  DmaEnt dma[8];
};

// describe the section's stage (DMA, FIRST, non-hoisted) loads
__device__ __forceinline__ void issuer_section(Issuer& I, const Prog& P, const LaunchParams& Pm, const Instr* sec,
                                               int n) {
  I.n_dma = 0;
  for (int i = 0; i < n && I.n_dma < 8; i++) {
    const Instr w = sec[i];
    if (w.op != OP_LD || (w.flags & (LF_DMA | LF_FIRST | LF_HOIST)) != (LF_DMA | LF_FIRST)) continue;
    const TensRec& T = P.tens[w.b];
    DmaEnt& e = I.dma[I.n_dma++];
    e.src = static_cast<const uint8_t*>(Pm.ptrs[T.binding]);
    e.vs0 = P.r == 2 ? T.vs[0] : 0;
    e.aux0 = w.aux0;
    e.esz = dtype_size(T.dtype);
    e.tens = w.b;
    if (w.flags & LF_COLV) e.kind = 0;
    else if (P.r == 2 && T.vs[0] == (int64_t)P.t_in) e.kind = 1;
    else if (P.r <= 2) e.kind = 2;
    else e.kind = 3;
  }
  I.stage_sec = I.n_dma > 0;
}

// one staged tile: arm the full barrier with the byte count, then issue the copies
__device__ __forceinline__ void issue_tile(const LaunchParams& Pm, const Prog& P, const Issuer& I, const TilePos& O,
                                           uint8_t* dst_base, uint64_t* bar) {
  const int o_in = O.oin;
  const int valid_in = min(P.t_in, P.n_in - o_in);
  const int nrows = P.r == 2 ? min(P.rows, P.n0 - O.od[0]) : 1;
  for (int mode = 0; mode < 2; mode++) {
    uint32_t total = 0;
    for (int k = 0; k < I.n_dma; k++) {
      const DmaEnt& e = I.dma[k];
      uint8_t* dst = dst_base + e.aux0;
      const uint32_t rowb = (uint32_t)(valid_in * e.esz);
      if (e.kind == 0) {  // one row shared by the tile (outer strides 0 within the tile)
        int64_t off = 0;
        bool ok = true;
        if (P.r > 2) ok = row_off_div(P.pr, P.r, O.od[0], O.od[1], O.od[2], 0, P.tens[e.tens].vs, &off);
        else off = (int64_t)O.od[0] * e.vs0;
        if (ok) {
          total += rowb;
          if (mode) bulk_g2s(dst, e.src + (off + o_in) * e.esz, rowb, bar);
        }
      } else if (e.kind == 1 && valid_in == P.t_in) {  // whole rows: one contiguous block
        const uint32_t bytes = (uint32_t)nrows * P.t_in * e.esz;
        total += bytes;
        if (mode) bulk_g2s(dst, e.src + ((int64_t)O.od[0] * e.vs0 + o_in) * e.esz, bytes, bar);
      } else if (e.kind <= 2) {  // rank <= 2, row by row
        const uint8_t* src = e.src + ((int64_t)O.od[0] * e.vs0 + o_in) * e.esz;
        total += rowb * nrows;
        if (mode)
          for (int row = 0; row < nrows; row++)
            bulk_g2s(dst + (size_t)row * P.t_in * e.esz, src + (int64_t)row * e.vs0 * e.esz, rowb, bar);
      } else {  // rank > 2
        for (int row = 0; row < P.rows; row++) {
          int64_t off;
          if (!row_off_div(P.pr, P.r, O.od[0], O.od[1], O.od[2], row, P.tens[e.tens].vs, &off)) continue;
          total += rowb;
          if (mode) bulk_g2s(dst + (size_t)row * P.t_in * e.esz, e.src + (off + o_in) * e.esz, rowb, bar);
        }
      }
    }
    if (mode == 0) mbar_arrive_expect_tx(bar, total);
  }
}

// Register slots.  ACC lives in registers (REG values per thread).  The addressable
// slots 1 and 2, and the scratch slot 3, live in per-thread shared-memory storage laid
// out [slot][q][thread] in float4 units (conflict-free), which keeps the interpreter
// loop's register state small enough for large tiles without spills.
__device__ __forceinline__ float4* slot_ptr(int k, int q) {
  return reinterpret_cast<float4*>(dvm_smem + kSlotOff) + ((k - 1) * (REG / 4) + q) * NTHREADS + threadIdx.x;
}
__device__ __forceinline__ void slot_read(int k, float (&x)[REG]) {
#pragma unroll
  for (int q = 0; q < REG / 4; q++) {
    const float4 f = *slot_ptr(k, q);
    x[4 * q] = f.x; x[4 * q + 1] = f.y; x[4 * q + 2] = f.z; x[4 * q + 3] = f.w;
  }
}
__device__ __forceinline__ void slot_write(int k, const float (&x)[REG]) {
#pragma unroll
  for (int q = 0; q < REG / 4; q++) *slot_ptr(k, q) = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
}

// ===================================================== consumer helpers ==
template <int VE>
struct Lanes {
  static constexpr int NV = REG / VE;  // vectors (segments) per thread per slot
  int row[NV];     // tile row of each vector
  int col[NV];     // first tile column of this lane's VE elements
  uint32_t seg;    // bit v: vector v maps to a segment of the tile
  uint32_t rowok;  // bit v: the segment's row lies inside the iteration space (per tile)
};

// fill the row-coordinate table of a rank > 2 program (all threads call it)
__device__ __forceinline__ void fill_rowcoords(const Prog& P) {
  if (P.r <= 2) return;
  __syncthreads();  // the previous program's tiles may still read the table
  for (int row = threadIdx.x; row < P.rows; row += NTHREADS) {
    int* rc = reinterpret_cast<int*>(dvm_smem + kRowCoordOff) + row * 4;
    int rr = row;
    for (int d = P.r - 2; d >= 0; d--) {
      const int td = (int)P.pr->t[d];
      rc[d] = rr % td;
      rr /= td;
    }
  }
  __syncthreads();
}

template <int VE>
__device__ __forceinline__ void lanes_for_prog(const Prog& P, int warp, int lane, Lanes<VE>& L) {
  const int a = VE * 32;
  L.seg = 0;
#pragma unroll
  for (int v = 0; v < Lanes<VE>::NV; v++) {
    const int s = v * NW + warp;
    if (s < P.segs) L.seg |= 1u << v;
    L.row[v] = s / P.m;
    L.col[v] = (s % P.m) * a + lane * VE;
  }
}

template <int VE>
__device__ __forceinline__ void lanes_for_tile(const Prog& P, const TilePos& O, Lanes<VE>& L) {
  uint32_t ok = 0;
#pragma unroll
  for (int v = 0; v < Lanes<VE>::NV; v++) {
    bool in = (L.seg >> v) & 1u;
    if (P.r == 2) {
      in = in && (O.od[0] + L.row[v] < P.n0);
    } else if (P.r > 2) {
      const int* rc = rowcoord(L.row[v]);
#pragma unroll
      for (int dd = 0; dd < 3; dd++)
        if (dd < P.r - 1) in = in && (O.od[dd] + rc[dd] < (int)P.pr->n[dd]);
    }
    if (in) ok |= 1u << v;
  }
  L.rowok = ok;
}

// valid elements of vector v among its VE (the inner tail of the last column tile)
template <int VE>
__device__ __forceinline__ int ncol(const Prog& P, const TilePos& O, const Lanes<VE>& L, int v) {
  const int nc = P.n_in - (O.oin + L.col[v]);
  return nc < 0 ? 0 : (nc > VE ? VE : nc);
}

// ---- loads into a register slot -------------------------------------------
template <int VE, int ESZ>
__device__ __forceinline__ void unpack(const uint8_t* p, float* dst) {
  if constexpr (ESZ == 4) {
#pragma unroll
    for (int q = 0; q < VE / 4; q++) {
      const float4 f = reinterpret_cast<const float4*>(p)[q];
      dst[4 * q] = f.x; dst[4 * q + 1] = f.y; dst[4 * q + 2] = f.z; dst[4 * q + 3] = f.w;
    }
  } else if constexpr (ESZ == 2) {
#pragma unroll
    for (int q = 0; q < VE / 8; q++) {
      const uint4 u = reinterpret_cast<const uint4*>(p)[q];
      dst[8 * q + 0] = bf16lo(u.x); dst[8 * q + 1] = bf16hi(u.x);
      dst[8 * q + 2] = bf16lo(u.y); dst[8 * q + 3] = bf16hi(u.y);
      dst[8 * q + 4] = bf16lo(u.z); dst[8 * q + 5] = bf16hi(u.z);
      dst[8 * q + 6] = bf16lo(u.w); dst[8 * q + 7] = bf16hi(u.w);
    }
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < VE; e++) dst[e] = (float)((w4[e / 4] >> (8 * (e % 4))) & 0xffu);
  }
}

__device__ __forceinline__ float load_scalar(const uint8_t* base, int64_t off, int dt) {
  if (dt == DT_F32) return __ldg(reinterpret_cast<const float*>(base) + off);
  if (dt == DT_BF16) return __uint_as_float(((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(base) + off)) << 16);
  return (float)__ldg(base + off);
}

// Hot paths are straight-line: the element size is resolved once per instruction, and
// per-vector validity turns into address clamping (shared memory) or a warp-uniform
// choice between a full-tile loop and a general masked loop (global memory).
template <int VE, int ESZ>
__device__ __forceinline__ void lds_vectors(float (&dst)[REG], const uint8_t* region, int rstride,
                                            const Lanes<VE>& L) {
#pragma unroll
  for (int v = 0; v < Lanes<VE>::NV; v++) {
    const bool in = (L.seg >> v) & 1u;
    const int eo = in ? (L.row[v] * rstride + L.col[v]) : 0;  // clamp: row 0, column 0 is inside
    unpack<VE, ESZ>(region + (size_t)eo * ESZ, dst + v * VE);
  }
}

template <int VE, int ESZ>
__device__ __forceinline__ void ldg_vectors_fast(float (&dst)[REG], const uint8_t* base, int64_t vs0, int oin,
                                                 const TilePos& O, const Lanes<VE>& L) {
  // rank <= 2, inner stride 1, every vector of the thread inside the tensor
#pragma unroll
  for (int v = 0; v < Lanes<VE>::NV; v++) {
    if (!((L.seg >> v) & 1u)) continue;
    const int64_t off = (int64_t)(O.od[0] + L.row[v]) * vs0 + oin + L.col[v];
    unpack<VE, ESZ>(base + off * ESZ, dst + v * VE);
  }
}

// LD of a FULL value into registers
// `scratch` is a slot whose contents are dead (used by the masked path)
template <int VE>
__device__ __forceinline__ void op_load(float (&dst)[REG], const Instr& w, const Prog& P, const Lanes<VE>& L,
                                        const TilePos& O, const LaunchParams& Pm, const uint8_t* stage_base,
                                        const uint8_t* hoist_base, int scratch) {
  constexpr int NV = Lanes<VE>::NV;
  const TensRec& T = P.tens[w.b];
  const int dt = T.dtype;
  if (w.flags & LF_DMA) {
    const uint8_t* region = ((w.flags & LF_HOIST) ? hoist_base + P.pr->hoist_base : stage_base) + w.aux0;
    const int rstride = (w.flags & LF_COLV) ? 0 : P.t_in;
    if (dt == DT_F32) {
      lds_vectors<VE, 4>(dst, region, rstride, L);
    } else if (dt == DT_BF16) {
      if constexpr (VE >= 8) lds_vectors<VE, 2>(dst, region, rstride, L);
    } else {
      if constexpr (VE == 16) lds_vectors<VE, 1>(dst, region, rstride, L);
    }
    return;
  }
  const uint8_t* base = static_cast<const uint8_t*>(Pm.ptrs[T.binding]);
  const int64_t vin = T.vs[P.r - 1];
  const int esz = dtype_size(dt);
  // full-tile fast path: every valid vector complete, rows inside, 16-byte aligned rows
  const bool mine = P.r <= 2 && vin == 1 && L.rowok == L.seg && O.oin + P.t_in <= P.n_in &&
                    (((P.r == 2 ? T.vs[0] : 0) * esz) & 15) == 0;
  if (__all_sync(0xffffffffu, mine)) {
    const int64_t vs0 = P.r == 2 ? T.vs[0] : 0;
    if (dt == DT_F32) {
      ldg_vectors_fast<VE, 4>(dst, base, vs0, O.oin, O, L);
    } else if (dt == DT_BF16) {
      if constexpr (VE >= 8) ldg_vectors_fast<VE, 2>(dst, base, vs0, O.oin, O, L);
    } else {
      if constexpr (VE == 16) ldg_vectors_fast<VE, 1>(dst, base, vs0, O.oin, O, L);
    }
    return;
  }
  // general masked path (ragged tails, strided views, rank > 2): a rolled loop through
  // the scratch slot keeps it compact
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* sc = reinterpret_cast<float*>(dvm_smem + kSlotOff) + (scratch - 1) * REG * NTHREADS;  // [q][thread][4]
#pragma unroll 1
  for (int j = 0; j < REG; j++) {
    const int v = j / VE, e = j % VE;
    const int sgi = v * NW + warp;
    const int row = sgi / P.m, col = (sgi % P.m) * (VE * 32) + lane * VE;
    float x = 0.f;
    int64_t off;
    if (sgi < P.segs && row_off(P, O, row, T.vs, off) && O.oin + col + e < P.n_in)
      x = load_scalar(base, off + (int64_t)(O.oin + col + e) * vin, dt);
    sc[((j >> 2) * NTHREADS + threadIdx.x) * 4 + (j & 3)] = x;
  }
  slot_read(scratch, dst);
}

// ---- stores from ACC --------------------------------------------------------
__device__ __forceinline__ void store_scalar(uint8_t* base, int64_t off, int dt, float x) {
  if (dt == DT_F32) reinterpret_cast<float*>(base)[off] = x;
  else if (dt == DT_BF16) reinterpret_cast<__nv_bfloat16*>(base)[off] = __float2bfloat16_rn(x);
  else base[off] = (uint8_t)(x != 0.f ? 1 : 0);
}

template <int VE, int ESZ>
__device__ __forceinline__ void pack_store(uint8_t* p, const float* s) {
  if constexpr (ESZ == 4) {
#pragma unroll
    for (int q = 0; q < VE / 4; q++)
      reinterpret_cast<float4*>(p)[q] = make_float4(s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3]);
  } else if constexpr (ESZ == 2) {
#pragma unroll
    for (int q = 0; q < VE / 8; q++) {
      uint4 u;
      u.x = pack_bf16(s[8 * q], s[8 * q + 1]);
      u.y = pack_bf16(s[8 * q + 2], s[8 * q + 3]);
      u.z = pack_bf16(s[8 * q + 4], s[8 * q + 5]);
      u.w = pack_bf16(s[8 * q + 6], s[8 * q + 7]);
      reinterpret_cast<uint4*>(p)[q] = u;
    }
  } else {
    uint32_t w4[4] = {0, 0, 0, 0};
#pragma unroll
    for (int e = 0; e < 16; e++) w4[e / 4] |= (uint32_t)(s[e] != 0.f ? 1 : 0) << (8 * (e % 4));
    *reinterpret_cast<uint4*>(p) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  }
}

template <int VE, int ESZ>
__device__ __forceinline__ void stg_vectors_fast(const float (&acc)[REG], uint8_t* base, int64_t vs0, int oin,
                                                 const TilePos& O, const Lanes<VE>& L) {
#pragma unroll
  for (int v = 0; v < Lanes<VE>::NV; v++) {
    if (!((L.seg >> v) & 1u)) continue;
    const int64_t off = (int64_t)(O.od[0] + L.row[v]) * vs0 + oin + L.col[v];
    pack_store<VE, ESZ>(base + off * ESZ, acc + v * VE);
  }
}

template <int VE>
__device__ __forceinline__ void op_store(const float (&acc)[REG], const Instr& w, const Prog& P, const Lanes<VE>& L,
                                         const TilePos& O, const LaunchParams& Pm) {
  constexpr int NV = Lanes<VE>::NV;
  const TensRec& T = P.tens[w.a];
  const int dt = T.dtype;
  const int esz = dtype_size(dt);
  uint8_t* base = static_cast<uint8_t*>(Pm.ptrs[T.binding]);
  const int64_t vin = T.vs[P.r - 1];
  const bool mine = P.r <= 2 && vin == 1 && L.rowok == L.seg && O.oin + P.t_in <= P.n_in &&
                    (((P.r == 2 ? T.vs[0] : 0) * esz) & 15) == 0;
  if (__all_sync(0xffffffffu, mine)) {
    const int64_t vs0 = P.r == 2 ? T.vs[0] : 0;
    if (dt == DT_F32) {
      stg_vectors_fast<VE, 4>(acc, base, vs0, O.oin, O, L);
    } else if (dt == DT_BF16) {
      if constexpr (VE >= 8) stg_vectors_fast<VE, 2>(acc, base, vs0, O.oin, O, L);
    } else {
      if constexpr (VE == 16) stg_vectors_fast<VE, 1>(acc, base, vs0, O.oin, O, L);
    }
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  slot_write(3, acc);
  const float* sc = reinterpret_cast<const float*>(dvm_smem + kSlotOff) + 2 * REG * NTHREADS;
#pragma unroll 1
  for (int j = 0; j < REG; j++) {
    const int v = j / VE, e = j % VE;
    const int sgi = v * NW + warp;
    const int row = sgi / P.m, col = (sgi % P.m) * (VE * 32) + lane * VE;
    int64_t off;
    if (sgi < P.segs && row_off(P, O, row, T.vs, off) && O.oin + col + e < P.n_in)
      store_scalar(base, off + (int64_t)(O.oin + col + e) * vin, dt, sc[((j >> 2) * NTHREADS + threadIdx.x) * 4 + (j & 3)]);
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

// powf with the exponents the normalisations use turned into cheaper exact-enough
// forms: x^-0.5 = 1/sqrt(x) (x = +-0 gives +inf as C99 pow does), x^1 = x, x^2 = x*x.
__device__ __forceinline__ float pow_fast(float a, float b) {
  if (b == -0.5f) return a == 0.f ? __int_as_float(0x7f800000) : 1.0f / sqrtf(a);
  if (b == 2.0f) return a * a;
  if (b == 1.0f) return a;
  return powf(a, b);
}

template <int OP>
__device__ __forceinline__ float bin(float a, float b) {
  if constexpr (OP == OP_ADD) return a + b;
  else if constexpr (OP == OP_SUB) return a - b;
  else if constexpr (OP == OP_MUL) return a * b;
  else if constexpr (OP == OP_DIV) return a / b;
  else if constexpr (OP == OP_MAX) return vmax(a, b);
  else if constexpr (OP == OP_MIN) return vmin(a, b);
  else return powf(a, b);
}
__device__ __forceinline__ float bin_rt(int op, float a, float b) {  // runtime opcode (row values)
  switch (op) {
    case OP_ADD: return a + b;
    case OP_SUB: return a - b;
    case OP_MUL: return a * b;
    case OP_DIV: return a / b;
    case OP_MAX: return vmax(a, b);
    case OP_MIN: return vmin(a, b);
    default: return pow_fast(a, b);
  }
}

// ACC (FULL) <- op(ACC, X) where X is a FULL value, a ROW buffer, or an immediate.
// The operand order is resolved outside the unrolled loops.
template <int OP>
__host__ __device__ constexpr bool commutative() { return OP == OP_ADD || OP == OP_MUL || OP == OP_MAX || OP == OP_MIN; }

template <int OP, bool REV>
__device__ __forceinline__ void bin_ff_(float (&acc)[REG], const float (&x)[REG]) {
#pragma unroll
  for (int e = 0; e < REG; e++) acc[e] = REV ? bin<OP>(x[e], acc[e]) : bin<OP>(acc[e], x[e]);
}
template <int OP>
__device__ __forceinline__ void bin_ff(float (&acc)[REG], const float (&x)[REG], bool rev) {
  if (!commutative<OP>() && rev) bin_ff_<OP, true>(acc, x);
  else bin_ff_<OP, false>(acc, x);
}
template <int OP, bool REV>
__device__ __forceinline__ void bin_fi_(float (&acc)[REG], float x) {
#pragma unroll
  for (int e = 0; e < REG; e++) acc[e] = REV ? bin<OP>(x, acc[e]) : bin<OP>(acc[e], x);
}
template <int OP>
__device__ __forceinline__ void bin_fi(float (&acc)[REG], float x, bool rev) {
  if (!commutative<OP>() && rev) bin_fi_<OP, true>(acc, x);
  else bin_fi_<OP, false>(acc, x);
}
// FULL op ROW(row buffer xrow) -> FULL
template <int VE, int OP, bool REV>
__device__ __forceinline__ void bin_fr_(float (&acc)[REG], const float* xrow, const Lanes<VE>& L) {
#pragma unroll
  for (int v = 0; v < Lanes<VE>::NV; v++) {
    const float x0 = xrow[L.row[v] & (kMaxRows - 1)];
#pragma unroll
    for (int e = 0; e < VE; e++) acc[v * VE + e] = REV ? bin<OP>(x0, acc[v * VE + e]) : bin<OP>(acc[v * VE + e], x0);
  }
}
template <int VE, int OP>
__device__ __forceinline__ void bin_fr(float (&acc)[REG], const float* xrow, const Lanes<VE>& L, bool rev) {
  if (!commutative<OP>() && rev) bin_fr_<VE, OP, true>(acc, xrow, L);
  else bin_fr_<VE, OP, false>(acc, xrow, L);
}
// ROW(row buffer arow) op FULL x -> FULL in ACC
template <int VE, int OP, bool REV>
__device__ __forceinline__ void bin_rf_(float (&acc)[REG], const float* arow, const float (&x)[REG],
                                        const Lanes<VE>& L) {
#pragma unroll
  for (int v = 0; v < Lanes<VE>::NV; v++) {
    const float a0 = arow[L.row[v] & (kMaxRows - 1)];
#pragma unroll
    for (int e = 0; e < VE; e++) acc[v * VE + e] = REV ? bin<OP>(x[v * VE + e], a0) : bin<OP>(a0, x[v * VE + e]);
  }
}
template <int VE, int OP>
__device__ __forceinline__ void bin_rf(float (&acc)[REG], const float* arow, const float (&x)[REG], const Lanes<VE>& L,
                                       bool rev) {
  if (!commutative<OP>() && rev) bin_rf_<VE, OP, true>(acc, arow, x, L);
  else bin_rf_<VE, OP, false>(acc, arow, x, L);
}

// warp-level all-reduce (xor butterfly: every lane ends with identical bits)
template <bool MAX>
__device__ __forceinline__ float warp_reduce(float p) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float q = __shfl_xor_sync(0xffffffffu, p, o);
    p = MAX ? vmax(p, q) : p + q;
  }
  return p;
}

// ---- the CTA's work ---------------------------------------------------------
// Shared-memory control state is addressed from dvm_smem with constant offsets so that
// no generic pointers occupy registers; only the ring geometry is kept in registers.
struct Ctl {
  int n_stages;
  uint32_t stage_bytes;
  uint32_t ring_off;   // byte offset of the stage ring in dvm_smem
  DevStatus st;
};
__device__ __forceinline__ uint64_t* bar_full(int s) { return reinterpret_cast<uint64_t*>(dvm_smem + kBarOff) + s; }
__device__ __forceinline__ uint64_t* bar_empty(int s) { return reinterpret_cast<uint64_t*>(dvm_smem + kBarOff) + 8 + s; }
__device__ __forceinline__ uint64_t* bar_hoist() { return reinterpret_cast<uint64_t*>(dvm_smem + kBarOff) + 16; }
__device__ __forceinline__ float* red_buf() { return reinterpret_cast<float*>(dvm_smem + kRedOff); }
__device__ __forceinline__ float* row_buf() { return reinterpret_cast<float*>(dvm_smem + kRowBufOff); }
__device__ __forceinline__ Issuer& issuer() { return *reinterpret_cast<Issuer*>(dvm_smem + kIssOff); }
__device__ __forceinline__ float* misc_scalar() { return reinterpret_cast<float*>(dvm_smem + kMiscOff); }
__device__ __forceinline__ volatile int* abort_flag() { return reinterpret_cast<volatile int*>(dvm_smem + kMiscOff + 16); }
__device__ __forceinline__ uint8_t* hoist_area() { return dvm_smem + kDataOff; }

// ---- heavy math -------------------------------------------------------------
// Transcendental and correctly rounded ops (sqrt, rsqrt, recip, log, exp, silu, div,
// pow) are long instruction sequences; unrolling them over the 16 register values in
// every operand form would make the interpreter's code far larger than the instruction
// caches.  They run instead as a rolled loop, 4 values per iteration, over the thread's
// scratch slot (slot 3) in shared memory: ACC is written there, transformed, and read
// back.  Light ops (add, sub, mul, max, min, abs, neg, floor, round, casts) stay
// unrolled in registers.
__device__ __forceinline__ bool heavy_unary(int op) {
  return op == OP_SQRT || op == OP_LOG || op == OP_EXP || op == OP_RSQRT || op == OP_RECIP || op == OP_SILU;
}

template <class F>
__device__ __forceinline__ float4 map4(float4 a, F f) {
  a.x = f(a.x); a.y = f(a.y); a.z = f(a.z); a.w = f(a.w);
  return a;
}

__device__ __forceinline__ void heavy_unary_loop(int op) {
  switch (op) {
#define DVM_HEAVY_U(OPC, EXPR)                                         \
  case OPC:                                                            \
    _Pragma("unroll 1") for (int q = 0; q < REG / 4; q++) {            \
      float4* p = slot_ptr(3, q);                                      \
      *p = map4(*p, [](float x) { return EXPR; });                     \
    }                                                                  \
    break;
    DVM_HEAVY_U(OP_SQRT, sqrtf(x))
    DVM_HEAVY_U(OP_RSQRT, 1.0f / sqrtf(x))
    DVM_HEAVY_U(OP_RECIP, 1.0f / x)
    DVM_HEAVY_U(OP_LOG, logf(x))
    DVM_HEAVY_U(OP_EXP, expf(x))
    DVM_HEAVY_U(OP_SILU, x / (1.0f + expf(-x)))
#undef DVM_HEAVY_U
    default: break;
  }
}

__device__ __forceinline__ float4 splat4(float v) { return make_float4(v, v, v, v); }

// ACC <- op(A, X) for DIV / POW (result FULL).  A is the scratch slot 3 (ACC written
// there) or, with arow, the ACC row buffer; X is an immediate (xslot < 0), ACC itself
// (xslot == 0), a slot (1, 2), or, with xrow != nullptr, a row buffer.
template <int VE>
__device__ __forceinline__ void heavy_binary_loop(int op, bool rev, bool arow, const float* xrow, int xslot, float xi,
                                                  int m) {
  const int warp = threadIdx.x >> 5;
  const float* RB = row_buf();
#pragma unroll 1
  for (int q = 0; q < REG / 4; q++) {
    int row = 0;
    if (arow || xrow) {  // the 4 values of iteration q lie in one segment (VE >= 4)
      const int v = (4 * q) / VE;
      row = ((v * NW + warp) / m) & (kMaxRows - 1);
    }
    float4* pa = slot_ptr(3, q);
    const float4 a = arow ? splat4(RB[row]) : *pa;
    const float4 x = xrow ? splat4(xrow[row]) : xslot > 0 ? *slot_ptr(xslot, q) : xslot == 0 ? a : splat4(xi);
    const float4 l = rev ? x : a, r = rev ? a : x;
    float4 o;
    if (op == OP_DIV) {
      o = make_float4(l.x / r.x, l.y / r.y, l.z / r.z, l.w / r.w);
    } else {
      o = make_float4(pow_fast(l.x, r.x), pow_fast(l.y, r.y), pow_fast(l.z, r.z), pow_fast(l.w, r.w));
    }
    *pa = o;
  }
}


// Thread 0: issue staged tiles of the current range until `limit` tiles are issued.
__device__ __forceinline__ void issue_upto(const LaunchParams& Pm, const uint8_t* img, const Ctl& C, int a,
                                           int limit, bool plain) {
  Issuer& I = issuer();
  while (I.issued < limit && !*abort_flag()) {
    if (plain) {
      while (true) {
        if (I.g >= I.g_end) return;
        const ProgRec* pr = reinterpret_cast<const ProgRec*>(img + sizeof(Header) + I.prog * sizeof(ProgRec));
        const int end = (int)(pr->tile_base + pr->block_dim);
        if (I.g >= end) {  // the current program is done: set up the next one
          I.prog++;
          Prog Q;
          load_prog(img, I.prog, Q, a);
          I.sec_off = (int)(Q.pr->body_off / sizeof(Instr)) + 1;
          I.sec_n = (int)Q.body[0].imm;
          issuer_section(I, Q, Pm, Q.body + 1, I.sec_n);
          I.tau = I.g - (int)Q.pr->tile_base;
          I.c0 = I.tau / Q.tiles_in;
          I.cin = I.tau - I.c0 * Q.tiles_in;
          continue;
        }
        if (!I.stage_sec) {  // nothing to stage in this program: skip its tiles
          I.g = end;
          continue;
        }
        break;
      }
    } else if (I.tau >= I.t_end || !I.stage_sec) {
      return;
    }
    Prog P;
    load_prog(img, I.prog, P, a);
    TilePos T;
    T.tau = I.tau;
    T.c0 = I.c0;
    T.cin = I.cin;
    pos_origin(P, T);
    const int stage = I.issued % C.n_stages;
    const uint32_t parity = ((I.issued / C.n_stages) & 1) ^ 1;
    if (!mbar_wait(bar_empty(stage), parity, C.st, abort_flag())) return;
    issue_tile(Pm, P, I, T, dvm_smem + C.ring_off + (size_t)stage * C.stage_bytes, bar_full(stage));
    I.issued++;
    I.tau++;
    if (++I.cin == P.tiles_in) {
      I.cin = 0;
      I.c0++;
    }
    if (plain) I.g++;
  }
}

// Element-wise op with opcode OPC on the accumulator, all operand forms.
#define DVM_BIN_CASE(OPC)                                               \
  case OPC:                                                             \
    if (imm) {                                                          \
      bin_fi<OPC>(R0, __uint_as_float(w.imm), rev);                     \
    } else if (ar) {                                                    \
      row_cross_read();                                                 \
      float X[REG];                                                     \
      slot_read(w.a, X);                                                \
      bin_rf<VE, OPC>(R0, RB, X, L, rev);                               \
    } else if (xr) {                                                    \
      row_cross_read();                                                 \
      bin_fr<VE, OPC>(R0, RB + w.a * kMaxRows, L, rev);                 \
    } else if (w.a == 0) {                                              \
      bin_ff<OPC>(R0, R0, rev);                                         \
    } else {                                                            \
      float X[REG];                                                     \
      slot_read(w.a, X);                                                \
      bin_ff<OPC>(R0, X, rev);                                          \
    }                                                                   \
    break;

// ROW-buffer loop: entry r belongs to thread r
#define DVM_ROWS_FOR(r) for (int r = threadIdx.x; r < P.rows; r += NTHREADS)

template <int VE>
__device__ __forceinline__ void exec_tile(const LaunchParams& Pm, const Prog& P, const Instr* body, int n,
                                          const TilePos& T, Lanes<VE>& L, int lane, int it, const Ctl& C,
                                          float& grand, float (&R0)[REG], bool& row_read, bool& row_dirty) {
  constexpr int NV = REG / VE;
  const TilePos& O = T;
  lanes_for_tile<VE>(P, O, L);
  const int stage = C.n_stages ? it % C.n_stages : 0;
  const uint32_t parity = C.n_stages ? (uint32_t)((it / C.n_stages) & 1) : 0;
  const uint8_t* stage_base = dvm_smem + C.ring_off + (size_t)stage * C.stage_bytes;
  const int warp = threadIdx.x >> 5;
  float* RB = row_buf();  // RB[k * kMaxRows + r]
  // Row buffers: entry r is written only by its owner thread (threadIdx.x == r) and
  // read either by the owner or by every thread (element-wise ops with a ROW operand).
  // A CTA barrier is needed before a cross-thread read that follows owner writes
  // (row_dirty), and before an owner write that follows cross-thread reads (row_read).
  auto row_write_begin = [&]() {
    if (row_read) {
      __syncthreads();
      row_read = false;
      row_dirty = false;
    }
  };
  auto row_write_end = [&]() { row_dirty = true; };
  auto row_cross_read = [&]() {
    if (row_dirty) {
      __syncthreads();
      row_dirty = false;
    }
    row_read = true;
  };
  for (int pc = 0; pc < n; pc++) {
    const Instr w = body[pc];
    const uint8_t fl = w.flags;
    switch (w.op) {
      case OP_WAIT:
        mbar_wait(bar_full(stage), parity, C.st, abort_flag());
        break;
      case OP_REL:
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty(stage));
        break;
      case OP_LD:
        if (fl & LF_ROWV) {
          // one value per tile row from a [.., 1]-shaped tensor
          row_write_begin();
          const TensRec& Tn = P.tens[w.b];
          const uint8_t* base = static_cast<const uint8_t*>(Pm.ptrs[Tn.binding]);
          float* dstrow = RB + w.a * kMaxRows;
          DVM_ROWS_FOR(r) {
            int64_t off;
            dstrow[r] = row_off(P, O, r, Tn.vs, off) ? load_scalar(base, off, Tn.dtype) : 0.f;
          }
          row_write_end();
        } else {
          // one load path into ACC; a load into a slot parks ACC in the scratch slot
          if (w.a != 0) slot_write(3, R0);
          op_load<VE>(R0, w, P, L, O, Pm, stage_base, hoist_area(), w.a != 0 ? (int)w.a : 3);
          if (w.a != 0) {
            slot_write(w.a, R0);
            slot_read(3, R0);
          }
        }
        break;
      case OP_ST:
        if (fl & LF_ROWV) {
          const TensRec& Tn = P.tens[w.a];
          uint8_t* base = static_cast<uint8_t*>(Pm.ptrs[Tn.binding]);
          DVM_ROWS_FOR(r) {
            int64_t off;
            if (row_off(P, O, r, Tn.vs, off)) store_scalar(base, off, Tn.dtype, RB[r]);
          }
        } else {
          op_store<VE>(R0, w, P, L, O, Pm);
        }
        break;
      case OP_MOV:
        if (fl & 1) {  // ROW value: copy between row buffers (owner threads)
          row_write_begin();
          DVM_ROWS_FOR(r) RB[w.a * kMaxRows + r] = RB[w.b * kMaxRows + r];
          row_write_end();
        } else if (w.a == 0) {
          if (w.b != 0) slot_read(w.b, R0);
        } else {
          slot_write(w.a, R0);
        }
        break;
      case OP_BCAST:
        row_cross_read();
#pragma unroll
        for (int v = 0; v < NV; v++) {
          const float x0 = RB[L.row[v] & (kMaxRows - 1)];
#pragma unroll
          for (int e = 0; e < VE; e++) R0[v * VE + e] = x0;
        }
        break;
      case OP_ADD: case OP_SUB: case OP_MUL: case OP_DIV: case OP_MAX: case OP_MIN: case OP_POW: {
        const bool rev = fl & CF_REV;
        const bool ar = fl & CF_AROW, xr = fl & CF_XROW, imm = fl & CF_IMM;
        if (ar && (xr || imm)) {
          // ROW op ROW -> ROW, in the ACC row buffer (owner threads)
          row_write_begin();
          const float xi = __uint_as_float(w.imm);
          const float* xrow = RB + w.a * kMaxRows;
          DVM_ROWS_FOR(r) {
            const float a0 = RB[r];
            const float x0 = imm ? xi : xrow[r];
            RB[r] = rev ? bin_rt(w.op, x0, a0) : bin_rt(w.op, a0, x0);
          }
          row_write_end();
          break;
        }
        if (w.op == OP_DIV || w.op == OP_POW) {
          if (ar || xr) row_cross_read();
          if (!ar) slot_write(3, R0);
          heavy_binary_loop<VE>(w.op, rev, ar, xr ? RB + w.a * kMaxRows : nullptr, imm ? -1 : (int)w.a,
                                __uint_as_float(w.imm), P.m);
          slot_read(3, R0);
          break;
        }
        switch (w.op) {
          DVM_BIN_CASE(OP_ADD) DVM_BIN_CASE(OP_SUB) DVM_BIN_CASE(OP_MUL)
          DVM_BIN_CASE(OP_MAX) DVM_BIN_CASE(OP_MIN)
          default: break;
        }
        break;
      }
      case OP_RSUM:
      case OP_RMAX: {
        // ACC (FULL) -> ACC row buffer.  Fixed order: each thread combines its vectors of
        // one row in order, the warp butterfly combines the lanes, then the row's owner
        // thread adds the warps' partials in warp order.
        const bool mx = w.op == OP_RMAX;
        const float ident = mx ? -INFINITY : 0.f;
        if (row_dirty || row_read) __syncthreads();  // red[] of an earlier reduction may still be read
        float run = ident;
#pragma unroll
        for (int v = 0; v < NV; v++) {
          if (!((L.seg >> v) & 1u)) continue;
          float p = ident;
          if ((L.rowok >> v) & 1u) {
            const int nc = ncol<VE>(P, O, L, v);
#pragma unroll
            for (int e = 0; e < VE; e++)
              if (e < nc) p = mx ? vmax(p, R0[v * VE + e]) : p + R0[v * VE + e];
          }
          run = mx ? vmax(run, p) : run + p;
          const bool last = v == NV - 1 || !((L.seg >> (v + 1)) & 1u) || L.row[v + 1] != L.row[v];
          if (last) {
            const float q = mx ? warp_reduce<true>(run) : warp_reduce<false>(run);
            if (lane == 0) red_buf()[L.row[v] * NW + warp] = q;
            run = ident;
          }
        }
        __syncthreads();
        DVM_ROWS_FOR(r) {
          const int nwc = P.m < NW ? P.m : NW;
          float q = ident;
          for (int j = 0; j < nwc; j++) {
            const float x = red_buf()[r * NW + ((r * P.m + j) % NW)];
            q = mx ? vmax(q, x) : q + x;
          }
          RB[r] = q;
        }
        row_read = false;
        row_dirty = true;
        break;
      }
      case OP_ASUM:
        if (fl & CF_AROW) {
          if (threadIdx.x < (unsigned)P.rows) {
            int64_t off;
            const int64_t zero4[4] = {0, 0, 0, 0};
            if (row_off(P, O, threadIdx.x, zero4, off)) grand += RB[threadIdx.x];
          }
        } else {
#pragma unroll
          for (int v = 0; v < NV; v++)
            if ((L.rowok >> v) & 1u) {
              const int nc = ncol<VE>(P, O, L, v);
#pragma unroll
              for (int e = 0; e < VE; e++)
                if (e < nc) grand += R0[v * VE + e];
            }
        }
        break;
      case OP_SQRT: case OP_ABS: case OP_LOG: case OP_EXP: case OP_ROUND: case OP_FLOOR:
      case OP_ISFIN: case OP_NEG: case OP_RSQRT: case OP_RECIP: case OP_SILU: case OP_CASTBF: {
        const int op = w.op;
        if (fl & CF_AROW) {
          row_write_begin();
          DVM_ROWS_FOR(r) RB[r] = unary_fn(op, RB[r]);
          row_write_end();
        } else if (heavy_unary(op)) {
          slot_write(3, R0);
          heavy_unary_loop(op);
          slot_read(3, R0);
        } else {
          switch (op) {  // light ops: one unrolled register loop per opcode
#define DVM_UNARY_CASE(OPC)                                                        \
  case OPC:                                                                        \
    _Pragma("unroll") for (int e = 0; e < REG; e++) R0[e] = unary_fn(OPC, R0[e]); \
    break;
            DVM_UNARY_CASE(OP_ABS) DVM_UNARY_CASE(OP_ROUND) DVM_UNARY_CASE(OP_FLOOR) DVM_UNARY_CASE(OP_ISFIN)
            DVM_UNARY_CASE(OP_NEG) DVM_UNARY_CASE(OP_CASTBF)
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
#undef DVM_ROWS_FOR
#undef DVM_BIN_CASE

// ---- grid-wide sum (GSUM) -------------------------------------------------
// Called by every thread of the CTA.  The result is identical on every CTA (fixed
// combination order).  The wait for the other CTAs is bounded; on expiry the status
// word is set and every thread of the CTA sees `abort`.
__device__ __forceinline__ float grid_sum(const LaunchParams& Pm, float grand, int lane) {
  const int warp = threadIdx.x >> 5;
  __syncthreads();
  const float p = warp_reduce<false>(grand);
  if (lane == 0) red_buf()[warp] = p;
  __syncthreads();
  if (threadIdx.x == 0) {
    float cta = 0.f;
    for (int w = 0; w < NW; w++) cta += red_buf()[w];
    Pm.partials[blockIdx.x] = cta;
    __threadfence();
    if (!(Pm.skip_arrival && blockIdx.x == 0)) atomicAdd(Pm.barrier, 1ull);
    const unsigned long long t0 = globaltimer();
    while (true) {
      const unsigned long long v = *reinterpret_cast<volatile unsigned long long*>(Pm.barrier);
      if (v >= Pm.barrier_target) break;
      if (globaltimer() - t0 > Pm.timeout_ns) {
        set_status(Pm.status, -100 /* DVM_E_TIMEOUT */);
        *abort_flag() = 1;
        break;
      }
      __nanosleep(256);
    }
    __threadfence();
  }
  __syncthreads();
  if (*abort_flag()) return 0.f;
  if (warp == 0) {
    float q = 0.f;
    for (int c = lane; c < (int)gridDim.x; c += 32) q += __ldcg(Pm.partials + c);
    q = warp_reduce<false>(q);
    if (lane == 0) *misc_scalar() = q;
  }
  __syncthreads();
  return *misc_scalar();
}

// ---- the kernel --------------------------------------------------------------
template <int VE>
__global__ void __launch_bounds__(NTHREADS, 1) vm_vec_kernel(const __grid_constant__ LaunchParams Pm) {
  uint8_t* smem = dvm_smem;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  {
    const uint32_t total = reinterpret_cast<const Header*>(Pm.image)->total_len;
    for (uint32_t i = tid * 16; i < total; i += NTHREADS * 16)
      *reinterpret_cast<uint4*>(smem + i) = *reinterpret_cast<const uint4*>(Pm.image + i);
  }
  const Header* H = reinterpret_cast<const Header*>(smem);
  Ctl C;
  if (tid == 0) {
    for (int s = 0; s < 8; s++) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), NW);
    }
    mbar_init(bar_hoist(), 1);
    *abort_flag() = 0;
    fence_mbar_init();
  }
  __syncthreads();
  C.n_stages = H->n_stages;
  C.stage_bytes = H->stage_bytes;
  C.ring_off = kDataOff + ((H->hoist_bytes + 127) & ~127u);
  C.st.word = Pm.status;
  C.st.limit_ns = Pm.timeout_ns;

  const int a = VE * 32;
  const int lo = blockIdx.x * (int)H->body_tile;
  const int hi = min(lo + (int)H->body_tile, (int)H->block_dim);
  const bool sectioned = reinterpret_cast<const ProgRec*>(smem + sizeof(Header))->kind == PK_SEC;
  const bool has_work = lo < hi;
  // a CTA without tiles leaves at once, except in a sectioned program, whose grid
  // barrier needs every CTA
  if (!has_work && !sectioned) return;
  const int n_progs = H->n_progs;

  // hoisted (tile-invariant) loads: once per CTA, all programs, one mbarrier phase
  if (tid == 0 && has_work) {
    uint32_t total = 0;
    TilePos O0;
    O0.tau = O0.c0 = O0.cin = 0;
    O0.od[0] = O0.od[1] = O0.od[2] = 0;
    O0.oin = 0;
    for (int mode = 0; mode < 2; mode++) {
      if (mode == 1) mbar_arrive_expect_tx(bar_hoist(), total);
      if (!H->hoist_bytes) continue;
      for (int p = 0; p < n_progs; p++) {
        Prog P;
        load_prog(smem, p, P, a);
        total += dma_tile(Pm, P, P.body, (int)P.pr->body_len, O0, hoist_area() + P.pr->hoist_base, bar_hoist(),
                          true, mode);
      }
    }
  }
  if (H->hoist_bytes && has_work) mbar_wait(bar_hoist(), 0, C.st, abort_flag());

  float R0[REG];
#pragma unroll
  for (int e = 0; e < REG; e++) R0[e] = 0.f;
  float grand = 0.f;
  bool row_read = false, row_dirty = false;
  int it = 0;  // staged tiles consumed
  Lanes<VE> L;
  Prog P;
  TilePos T;

  // One walk over the CTA's work, with a single tile-execution site:
  //   plain/stacked — the concatenated tile range [lo, hi) across programs;
  //   sectioned     — the top-level control flow (TILES / GSUM / SST / JLE0 / JMP / END).
  int p = -1;        // plain: current program
  int g = lo;        // plain: next concatenated tile
  int pc = 0;        // sectioned: next top-level instruction
  int tau = 0, t_end = 0;
  const Instr* sec = nullptr;
  int sec_n = 0;
  bool staged = false;
  float S = 0.f;
  if (sectioned) {
    p = 0;
    load_prog(smem, 0, P, a);
    lanes_for_prog<VE>(P, warp, lane, L);
    fill_rowcoords(P);
  }
  while (true) {
    if (!sectioned) {
      if (g >= hi) break;
      if (p < 0 || g >= (int)(P.pr->tile_base + P.pr->block_dim)) {
        p++;
        while (g >= (int)(reinterpret_cast<const ProgRec*>(smem + sizeof(Header) + p * sizeof(ProgRec))->tile_base +
                          reinterpret_cast<const ProgRec*>(smem + sizeof(Header) + p * sizeof(ProgRec))->block_dim))
          p++;
        load_prog(smem, p, P, a);
        lanes_for_prog<VE>(P, warp, lane, L);
        fill_rowcoords(P);
        sec = P.body + 1;
        sec_n = (int)P.body[0].imm;
        staged = section_has_stage(sec, sec_n);
        tau = g - (int)P.pr->tile_base;
        pos_start(P, T, tau);
        if (tid == 0 && it == 0) {
          Issuer& I = issuer();
          I.prog = p;
          I.g = g;
          I.g_end = hi;
          I.sec_off = (int)(P.pr->body_off / sizeof(Instr)) + 1;
          I.sec_n = sec_n;
          issuer_section(I, P, Pm, sec, sec_n);
          I.tau = tau;
          I.c0 = T.c0;
          I.cin = T.cin;
          I.issued = 0;
          issue_upto(Pm, smem, C, a, C.n_stages ? C.n_stages - 1 : 0, true);
        }
      }
    } else {
      bool done = false;
      while (tau >= t_end) {
        if (pc >= (int)P.pr->body_len) {
          done = true;
          break;
        }
        const Instr w = P.body[pc];
        if (w.op == OP_TILES) {
          sec = P.body + pc + 1;
          sec_n = (int)w.imm;
          staged = section_has_stage(sec, sec_n);
          tau = lo;
          t_end = min(hi, (int)P.pr->block_dim);
          pc += 1 + sec_n;
          if (tau < t_end) {
            pos_start(P, T, tau);
            if (tid == 0 && staged) {
              Issuer& I = issuer();
              I.prog = 0;
              I.sec_off = (int)(P.pr->body_off / sizeof(Instr)) + (int)(sec - P.body);
              I.sec_n = sec_n;
              issuer_section(I, P, Pm, sec, sec_n);
              I.tau = tau;
              I.t_end = t_end;
              I.c0 = T.c0;
              I.cin = T.cin;
              I.issued = it;
              issue_upto(Pm, smem, C, a, it + C.n_stages - 1, false);
            }
          }
        } else if (w.op == OP_GSUM) {
          S = grid_sum(Pm, grand, lane);
          row_read = row_dirty = false;
          if (*abort_flag()) {
            done = true;
            break;
          }
          pc++;
        } else if (w.op == OP_SST) {
          if (blockIdx.x == 0 && tid == 0) {
            const TensRec& Tn = P.tens[w.a];
            store_scalar(static_cast<uint8_t*>(Pm.ptrs[Tn.binding]), 0, Tn.dtype, S);
          }
          pc++;
        } else if (w.op == OP_JLE0) {
          pc += 1 + (S > 0.f ? 0 : (int)w.imm);
        } else if (w.op == OP_JMP) {
          pc += 1 + (int)w.imm;
        } else {
          done = true;  // END
          break;
        }
      }
      if (done) break;
    }
    if (staged && tid == 0) issue_upto(Pm, smem, C, a, it + C.n_stages, !sectioned);
    exec_tile<VE>(Pm, P, sec, sec_n, T, L, lane, it, C, grand, R0, row_read, row_dirty);
    if (staged) it++;
    pos_next(P, T);
    if (sectioned) tau++;
    else g++;
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
