"""Write tests/golden/*.txt: reference launch images, one shape per workload.

Run from the repository root:  python -m oracle.make_golden
Uses only the oracle package (reference encoder) and the workload op lists.  Each file
records the op stream, the input shapes and the encoded bytes as hex, so that a change
to the bytecode format or to the tiling/lowering rules shows up as a diff.  The format
follows the bytecode specification (code header with block_dim / body_tile / kernel
type and a code body with inserted syncs, review page sections 4.2-4.3; instructions of
Table 1, section 4.1).
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import ref_encoder as R  # noqa: E402
from bytecode_vm_jit_gb300 import workloads as W  # noqa: E402

CASES = {
    "sqrt_add_4096x1024": (W.SQRT_ADD_OPS, {"a": ("f32", (4096, 1024), None), "b": ("f32", (4096, 1024), None)}, W.SQRT_ADD_OUT),
    "layernorm_r1000": (W.LAYERNORM_OPS, {"x": ("f32", (1000, 4096), None), "gamma": ("f32", (4096,), None),
                                          "beta": ("f32", (4096,), None)}, W.LAYERNORM_OUT),
    "layernorm_r1": (W.LAYERNORM_OPS, {"x": ("f32", (1, 4096), None), "gamma": ("f32", (4096,), None),
                                       "beta": ("f32", (4096,), None)}, W.LAYERNORM_OUT),
    "if_else_add_t300": (W.IF_ELSE_ADD_OPS, {"x": ("bf16", (300, 8192), None), "z": ("bf16", (300, 8192), None)}, W.IF_ELSE_ADD_OUT),
    "matmul_abs_m100": (W.MATMUL_ABS_OPS, {"A": ("bf16", (100, 4096), None), "W": ("bf16", (4096, 4096), [1, 4096]),
                                           "bias": ("bf16", (4096,), None)}, W.MATMUL_ABS_OUT),
    "matmul_abs_m8192": (W.MATMUL_ABS_OPS, {"A": ("bf16", (8192, 4096), None), "W": ("bf16", (4096, 4096), [1, 4096]),
                                            "bias": ("bf16", (4096,), None)}, W.MATMUL_ABS_OUT),
    "qwen_step_t200": (W.QWEN_STEP_OPS, {"x": ("bf16", (200, 5120), None), "r": ("bf16", (200, 5120), None),
                                         "w": ("bf16", (5120,), None), "g": ("bf16", (200, 17408), None),
                                         "u": ("bf16", (200, 17408), None)}, W.QWEN_STEP_OUT),
}


def render(name):
    ops, inputs, outs = CASES[name]
    _, _, launches = R.replay(ops, inputs, outs)
    lines = ["# golden launch images for %s (written by oracle/make_golden.py)" % name,
             "# inputs: " + "; ".join("%s %s %s strides=%s" % (k, v[0], list(v[1]), v[2]) for k, v in inputs.items()),
             "# device: " + " ".join("%s=%d" % kv for kv in sorted(R.DEFAULT_DESC.items()))]
    for i, (img, binds) in enumerate(launches):
        lines.append("launch %d bindings %s" % (i, " ".join(str(b) for b in binds)))
        for o in range(0, len(img), 32):
            lines.append(img[o:o + 32].hex())
    return "\n".join(lines) + "\n"


def main():
    out = os.path.join(ROOT, "tests", "golden")
    os.makedirs(out, exist_ok=True)
    for name in CASES:
        with open(os.path.join(out, name + ".txt"), "w") as f:
            f.write(render(name))
        print("wrote", name)


if __name__ == "__main__":
    main()
