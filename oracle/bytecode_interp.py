"""Plain numpy interpreter of DVM launch images (test infrastructure only).

Executes a launch image the way the review page's VM algorithm describes it
(section 4.4): the tiles of the launch are split into contiguous per-core ranges of
body_tile tiles; for each tile the body is decoded instruction by instruction and the
matching virtual-instruction function runs.  Registers hold whole tiles as numpy
arrays in fp64 that are rounded to float32 after every instruction (the interpreter
models fp32 registers); a ROW value is one column per tile row.

It decodes the byte layout of the bytecode specification independently of both
encoders, so running an encoded program here and comparing with the op-graph
evaluator checks the lowering (slot use, operand order, row/full kinds, syncs,
sections and jumps) without a GPU.
"""
import struct

import numpy as np

from .bf16 import round_bf16, bf16_bits_to_f64

ESZ = {1: 4, 2: 2, 3: 1}


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def _imm(u):
    return struct.unpack("<f", struct.pack("<I", u))[0]


UNARY = {
    0x10: np.sqrt, 0x11: np.abs, 0x12: np.log, 0x13: np.exp, 0x14: np.rint,
    0x15: np.floor, 0x16: lambda x: np.isfinite(x).astype(np.float64), 0x17: np.negative,
    0x18: lambda x: 1.0 / np.sqrt(x), 0x19: lambda x: 1.0 / x,
    0x1A: lambda x: x / (1.0 + np.exp(-x)), 0x1B: round_bf16,
}
BINARY = {0x20: np.add, 0x21: np.subtract, 0x22: np.multiply, 0x23: np.divide,
          0x24: np.maximum, 0x25: np.minimum, 0x26: np.power}


class Tensor:
    """A bound buffer: flat fp64 storage (values) + dtype; element offsets index it."""

    def __init__(self, flat, dtype):
        self.flat, self.dtype = flat, dtype


def parse(img):
    h = struct.unpack_from("<IHBBIHHIIIBBHIIII", img, 0)
    hdr = dict(magic=h[0], version=h[1], kernel_type=h[2], flags=h[3], total=h[4],
               n_progs=h[5], n_bind=h[6], grid=h[7], block_dim=h[8], body_tile=h[9],
               ve=h[10], n_stages=h[11], n_slots=h[12], stage_bytes=h[13], hoist_bytes=h[14])
    progs = []
    for p in range(hdr["n_progs"]):
        r = struct.unpack_from("<IIBBBBIII4I4III", img, 48 + 64 * p)
        prog = dict(block_dim=r[0], tile_base=r[1], rank=r[2], n_tens=r[3], kind=r[4],
                    body_off=r[6], body_len=r[7], tens_off=r[8], n=list(r[9:13]),
                    t=list(r[13:17]), K=r[17], hoist_base=r[18])
        tens = []
        for i in range(prog["n_tens"]):
            e = struct.unpack_from("<BBHI4q", img, prog["tens_off"] + 40 * i)
            tens.append(dict(dtype=e[0], binding=e[1], vs=list(e[4:8])))
        prog["tensors"] = tens
        body = []
        for i in range(prog["body_len"]):
            w = struct.unpack_from("<BBBBIII", img, prog["body_off"] + 16 * i)
            body.append(dict(op=w[0], a=w[1], b=w[2], flags=w[3], imm=w[4], aux0=w[5]))
        prog["body"] = body
        progs.append(prog)
    return hdr, progs


class Interp:
    def __init__(self, img, buffers):
        """buffers: list (binding order) of (flat fp64 numpy array, dtype code)."""
        self.hdr, self.progs = parse(img)
        self.buf = [Tensor(np.asarray(b, dtype=np.float64).reshape(-1), dt) for b, dt in buffers]

    # -- tile geometry
    def tile_index_grid(self, prog, tau):
        r = prog["rank"]
        n, t = prog["n"][:r], prog["t"][:r]
        tiles = [-(-n[d] // t[d]) for d in range(r)]
        coords = []
        rem = tau
        for d in reversed(range(r)):
            coords.append(rem % tiles[d])
            rem //= tiles[d]
        coords = list(reversed(coords))
        origin = [coords[d] * t[d] for d in range(r)]
        rows = 1
        for d in range(r - 1):
            rows *= t[d]
        # outer coordinates of each tile row
        idx = np.zeros((rows, r - 1), dtype=np.int64)
        for rho in range(rows):
            rr = rho
            for d in reversed(range(r - 1)):
                idx[rho, d] = origin[d] + rr % t[d]
                rr //= t[d]
        cols = origin[r - 1] + np.arange(t[r - 1])
        rvalid = np.all(idx < np.array(n[:r - 1]), axis=1) if r > 1 else np.ones(rows, bool)
        cvalid = cols < n[r - 1]
        return idx, cols, rvalid, cvalid

    def offsets(self, ten, idx, cols, rowv):
        vs = ten["vs"]
        r = len(idx[0]) + 1 if len(idx) else 1
        base = np.zeros(idx.shape[0], dtype=np.int64)
        for d in range(idx.shape[1]):
            base += idx[:, d] * vs[d]
        if rowv:
            return base[:, None]
        return base[:, None] + cols[None, :] * vs[idx.shape[1]]

    def load(self, prog, ti, idx, cols, mask, rowv):
        ten = prog["tensors"][ti]
        b = self.buf[ten["binding"]]
        off = self.offsets(ten, idx, cols, rowv)
        m = mask[:, :1] if rowv else mask
        vals = np.zeros(off.shape)
        vals[m] = b.flat[off[m]]
        return vals

    def store(self, prog, ti, idx, cols, mask, val, rowv):
        ten = prog["tensors"][ti]
        b = self.buf[ten["binding"]]
        v = val
        if ten["dtype"] == 2:
            v = round_bf16(v)
        elif ten["dtype"] == 1:
            v = _f32(v)
        off = self.offsets(ten, idx, cols, rowv)
        m = mask[:, :1] if rowv else mask
        vv = np.broadcast_to(v, off.shape)
        b.flat[off[m]] = vv[m]

    # -- execution
    def run(self):
        hdr = self.hdr
        progs = self.progs
        if hdr["kernel_type"] == 2:
            for prog in progs:
                self.run_cube(prog)
            return
        if len(progs) == 1 and progs[0]["kind"] == 1:
            self.run_sectioned(progs[0])
            return
        # stacked: concatenated tile space, contiguous per-core ranges
        for core in range(hdr["grid"]):
            lo = core * hdr["body_tile"]
            hi = min(lo + hdr["body_tile"], hdr["block_dim"])
            for g in range(lo, hi):
                for prog in progs:
                    if prog["tile_base"] <= g < prog["tile_base"] + prog["block_dim"]:
                        body = prog["body"][1:1 + prog["body"][0]["imm"]]
                        self.exec_tile(prog, g - prog["tile_base"], body, {})

    def run_sectioned(self, prog):
        hdr = self.hdr
        body = prog["body"]
        pc = 0
        grand = [0.0]
        S = None
        while True:
            w = body[pc]
            op = w["op"]
            if op == 0x40:
                n = w["imm"]
                sec = body[pc + 1:pc + 1 + n]
                for core in range(hdr["grid"]):
                    lo = core * hdr["body_tile"]
                    hi = min(lo + hdr["body_tile"], prog["block_dim"])
                    for tau in range(lo, hi):
                        self.exec_tile(prog, tau, sec, {"grand": grand})
                pc += 1 + n
            elif op == 0x41:
                S = float(np.float32(grand[0]))
                pc += 1
            elif op == 0x44:
                ten = prog["tensors"][w["a"]]
                b = self.buf[ten["binding"]]
                b.flat[0] = round_bf16(S) if ten["dtype"] == 2 else _f32(S)
                pc += 1
            elif op == 0x42:
                pc += 1 + (0 if S > 0 else _s32(w["imm"]))
            elif op == 0x43:
                pc += 1 + _s32(w["imm"])
            elif op == 0x45:
                return
            else:
                raise ValueError("opcode %#x at top level" % op)

    def exec_tile(self, prog, tau, body, state):
        idx, cols, rvalid, cvalid = self.tile_index_grid(prog, tau)
        mask = rvalid[:, None] & cvalid[None, :]
        R = {}
        kind = {}
        with np.errstate(all="ignore"):
            for w in body:
                op = w["op"]
                if op in (0x05, 0x06):
                    continue
                if op == 0x01:
                    rowv = bool(w["flags"] & 8)
                    R[w["a"]] = _f32(self.load(prog, w["b"], idx, cols, mask, rowv))
                    kind[w["a"]] = "ROW" if rowv else "FULL"
                elif op == 0x02:
                    self.store(prog, w["a"], idx, cols, mask, R[0], bool(w["flags"] & 8))
                elif op == 0x03:
                    R[w["a"]] = R[w["b"]]
                    kind[w["a"]] = kind[w["b"]]
                elif op == 0x04:
                    R[0] = np.broadcast_to(R[0], mask.shape).copy()
                    kind[0] = "FULL"
                elif op in UNARY:
                    R[0] = _f32(UNARY[op](R[0]))
                elif op in BINARY:
                    x = _imm(w["imm"]) if w["flags"] & 8 else R[w["a"]]
                    if w["flags"] & 4:
                        res = BINARY[op](x, R[0])
                    else:
                        res = BINARY[op](R[0], x)
                    if not (w["flags"] & 8) and kind.get(w["a"]) == "FULL":
                        kind[0] = "FULL"
                    R[0] = _f32(res)
                elif op in (0x30, 0x31):
                    v = np.where(mask, R[0], 0.0 if op == 0x30 else -np.inf)
                    R[0] = _f32(np.sum(v, axis=1, keepdims=True) if op == 0x30 else np.max(v, axis=1, keepdims=True))
                    kind[0] = "ROW"
                elif op == 0x32:
                    m = mask if R[0].shape[1] > 1 else rvalid[:, None]
                    state["grand"][0] += float(np.sum(np.where(m, R[0], 0.0)))
                elif op == 0x50:
                    R[0] = self.mma_tile(prog, w, idx, cols, mask)
                    kind[0] = "FULL"
                else:
                    raise ValueError("opcode %#x in a tile body" % op)

    def mma_tile(self, prog, w, idx, cols, mask):
        ta, tw = prog["tensors"][w["a"]], prog["tensors"][w["b"]]
        A, Wb = self.buf[ta["binding"]], self.buf[tw["binding"]]
        K = prog["K"]
        rows = idx[:, 0]
        kk = np.arange(K)
        rv = np.minimum(rows, prog["n"][0] - 1)
        cv = np.minimum(cols, prog["n"][1] - 1)
        a = A.flat[rv[:, None] * ta["vs"][0] + kk[None, :] * ta["vs"][1]]
        wm = Wb.flat[kk[:, None] * tw["vs"][0] + cv[None, :] * tw["vs"][1]]
        return _f32(a @ wm)

    def run_cube(self, prog):
        # K-split tiles of one output block together compute the block's full product:
        # each output block is evaluated once, over all of K
        ks = -(-prog["K"] // prog["t"][2])
        for tau in range(prog["block_dim"] // ks):
            self.exec_tile(prog, tau, prog["body"][1:1 + prog["body"][0]["imm"]], {})


def _s32(u):
    return u - (1 << 32) if u >= (1 << 31) else u


def run_image(img, bindings):
    """bindings: list of (flat fp64 array, dtype code) in binding order; outputs are
    written in place into the arrays."""
    it = Interp(img, bindings)
    it.run()
    return [t.flat for t in it.buf]
