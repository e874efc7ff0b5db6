"""Source checks of the CUDA kernels that the launch mode relies on.

Every kernel of the library is launched with programmatic stream
serialization, so it may start while the kernel before it in the stream is
still running.  That is safe only if each kernel calls grid_dep_wait() in
every CTA before it touches global memory.  A kernel added without the wait,
or launched another way, would race silently; these checks fail instead."""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "diffusion_transformer_image_gb300", "csrc")


def sources():
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh")):
            yield f, re.sub(r"//[^\n]*", "", open(os.path.join(CSRC, f)).read())


def kernel_bodies():
    """(file, kernel name, body) of every __global__ function."""
    for f, src in sources():
        for m in re.finditer(r"__global__\s+void\s+(?:__launch_bounds__\([^)]*\)\s*)?(\w+)\s*\(", src):
            i, depth = m.end() - 1, 0
            while True:   # the parameter list
                depth += {"(": 1, ")": -1}.get(src[i], 0)
                if depth == 0:
                    break
                i += 1
            start = src.index("{", i)
            j, depth = start, 0
            while True:   # the body
                depth += {"{": 1, "}": -1}.get(src[j], 0)
                if depth == 0:
                    break
                j += 1
            yield f, m.group(1), src[start:j + 1]


def test_every_kernel_waits_for_its_predecessor():
    kernels = list(kernel_bodies())
    assert len(kernels) >= 15
    for f, name, body in kernels:
        assert "grid_dep_wait();" in body, f"{f}: {name} never waits for the kernel before it"
        assert body.index("grid_dep_wait();") < body.index("grid_dep_launch();"), (f, name)


def test_global_accesses_follow_the_wait_in_simple_kernels():
    # kernels without a set-up phase wait first thing, before any statement
    # that could read or write global memory
    for f, name, body in kernel_bodies():
        stmts = [s.strip() for s in body[1:].split(";") if s.strip()]
        if name in ("gemm_kernel", "attn_kernel", "rotq_tma_kernel", "ln_rotq_tma_kernel"):
            continue   # set-up (barriers, tensor memory) first; checked by review
        head = [s for s in stmts[:3] if not s.startswith("__shared__") and not s.startswith("extern")]
        assert head and head[0].startswith("grid_dep_wait()"), (f, name, stmts[:3])


def test_every_launch_goes_through_launch_k():
    for f, src in sources():
        assert "<<<" not in src, f"{f}: a launch bypasses launch_k"
        if f != "internal.h":
            assert "cudaLaunchKernelEx" not in src, f"{f}: a launch bypasses launch_k"
