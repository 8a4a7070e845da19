"""Source checks of the launch contract every libzc kernel relies on (no GPU).

Every kernel is launched as a programmatic dependent launch, so it may start
while the kernel before it on the stream is still running; stream order for
data holds only because each thread executes griddepcontrol.wait (pdl_wait(),
or pdl_begin(), which also lets the next launch be scheduled) before it
touches global memory.  A kernel may first set up shared memory (mbarriers,
tables, cleared bins), which then overlaps the end of the previous kernel.
These checks keep that true for every kernel in csrc/: each __global__
function lets the next launch be scheduled among its first statements, and
the source before its first wait names no global access (no launch
parameters other than plain flags such as p.single, no loads, atomics or bulk
copies); and no kernel is launched with
the triple-chevron syntax (which would bypass launch_kernel and its
attributes).
"""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "lossless_bf16_exponent_zc_gb300",
                    "csrc")


def _sources():
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(CSRC, name)) as f:
                yield name, f.read()


def _kernels(text):
    """(name, body) of each __global__ function definition."""
    for m in re.finditer(r"__global__\s+void\s+(?:__launch_bounds__\([^)]*\)\s+)?(\w+)\s*\(", text):
        brace = text.index("{", m.end())
        depth, i = 0, brace
        while True:
            if text[i] == "{":
                depth += 1
            elif text[i] == "}":
                depth -= 1
                if depth == 0:
                    break
            i += 1
        yield m.group(1), text[brace + 1:i]


def test_every_kernel_waits_for_its_predecessor_first():
    found = 0
    for name, text in _sources():
        for kernel, body in _kernels(text):
            found += 1
            code = re.sub(r"//.*", "", body)
            statements = [s.strip() for s in code.split(";") if s.strip()]
            head = statements[:8]  # shared-memory addresses may be computed first
            assert any(s.endswith(("pdl_begin()", "pdl_allow_dependents()")) for s in head), \
                f"{name}: {kernel} does not let the next launch be scheduled first"
            waits = [i for i in (code.find("pdl_begin()"), code.find("pdl_wait()")) if i >= 0]
            assert waits, f"{name}: {kernel} never waits for the previous grid"
            before = code[:min(waits)]
            # nothing before the wait may touch global memory
            assert not re.search(r"\bp\.(?!single\b)|__ldg|ld_relaxed|st_relaxed|atomic|tma_|cp_async|\bws->|\bin\s*[\[+]|launch_epoch|launch_hold",
                                 before), f"{name}: {kernel} may access global memory before its wait"
    assert found >= 7  # encode (with its raw bypass), decode, reduce, histogram, pipeline link, QLC encode and decode


def test_no_triple_chevron_launches():
    for name, text in _sources():
        code = re.sub(r"//.*", "", text)
        assert "<<<" not in code, f"{name} launches a kernel without launch_kernel()"


def test_launch_kernel_sets_programmatic_serialization():
    with open(os.path.join(CSRC, "zc_api.cu")) as f:
        api = f.read()
    body = api[api.index("cudaError_t launch_kernel("):]
    body = body[:body.index("\n}\n")]
    assert "cudaLaunchAttributeProgrammaticStreamSerialization" in body
    assert "programmaticStreamSerializationAllowed = 1" in body
    assert "cudaLaunchKernelExC" in body
