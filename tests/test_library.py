"""Host-side checks of the C-ABI library: it loads without a GPU, exports every
function include/ra.h declares, and rejects invalid requests before touching
the device (no compute call is made here)."""
import ctypes
import os

import pytest

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import binding as rb


def test_library_exports_every_declared_symbol():
    L = ra.lib()
    names = rb.header_functions()
    assert {"ra_forward", "ra_forward_f32", "ra_forward_ws", "ra_workspace_bytes", "ra_permute",
            "ra_merge", "ra_check", "ra_status_string", "ra_version",
            "ra_schedule_stats"} <= set(names)
    for n in names:
        assert getattr(L, n) is not None


def test_status_strings_and_version():
    assert ra.status_string(0) == "RA_OK"
    assert ra.status_string(1) == "RA_ERR_INVALID_ARG"
    assert ra.status_string(5) == "RA_ERR_TIMEOUT"
    assert ra.status_string(99) == "RA_ERR_UNKNOWN"
    assert "sm_103a" in ra.version()


# Fake, 16-byte aligned, non-overlapping "device" addresses: validation runs
# on the host and must reject these requests before any CUDA call.
Q, K, V, OUT, LSE = (ctypes.c_void_p(0x10000000 * (i + 1)) for i in range(5))


def _fwd(B=1, H=4, Hkv=2, S=256, d=128, N=2, layout=0, causal=1, q=Q, out=OUT, lse=LSE):
    return ra.lib().ra_forward(q, K, V, out, lse, B, H, Hkv, S, d, N, layout, causal, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(B=0), rb.RA_ERR_INVALID_ARG),
    (dict(H=3), rb.RA_ERR_INVALID_ARG),            # H % Hkv != 0
    (dict(S=255), rb.RA_ERR_INVALID_ARG),          # S % n_blocks != 0
    (dict(N=0), rb.RA_ERR_INVALID_ARG),
    (dict(layout=2), rb.RA_ERR_INVALID_ARG),
    (dict(causal=3), rb.RA_ERR_INVALID_ARG),
    (dict(d=96), rb.RA_ERR_UNSUPPORTED),           # tensor-core path: d in {64, 128}
    (dict(q=ctypes.c_void_p(0x10000008)), rb.RA_ERR_INVALID_ARG),  # misaligned
    (dict(q=ctypes.c_void_p(0)), rb.RA_ERR_INVALID_ARG),           # null
    (dict(out=ctypes.c_void_p(0x10000000 + 4096)), rb.RA_ERR_INVALID_ARG),  # out overlaps q
    (dict(lse=ctypes.c_void_p(0x40000000 + 64)), rb.RA_ERR_INVALID_ARG),   # lse overlaps out
])
def test_forward_rejects_invalid_requests(kw, expect):
    assert _fwd(**kw) == expect


def test_f32_and_ws_validation():
    L = ra.lib()
    assert L.ra_forward_f32(Q, K, V, OUT, LSE, 1, 1, 1, 32, 300, 4, 0, 0, None) == rb.RA_ERR_UNSUPPORTED
    assert L.ra_forward_f32(Q, K, V, OUT, LSE, 1, 1, 1, 30, 16, 4, 0, 0, None) == rb.RA_ERR_INVALID_ARG
    # striped needs a workspace: null workspace is rejected before any launch
    assert L.ra_forward_ws(Q, K, V, OUT, LSE, 1, 4, 2, 256, 128, 2, 1, 1, 0, 0, None, 0,
                           None) == rb.RA_ERR_WORKSPACE
    # misaligned workspace
    assert L.ra_forward_ws(Q, K, V, OUT, LSE, 1, 4, 2, 256, 128, 2, 1, 1, 0, 0,
                           ctypes.c_void_p(0x50000010), 1 << 30, None) == rb.RA_ERR_WORKSPACE
    # bad mode / dtype
    assert L.ra_forward_ws(Q, K, V, OUT, LSE, 1, 4, 2, 256, 128, 2, 0, 1, 0, 7, None, 0,
                           None) == rb.RA_ERR_INVALID_ARG
    assert L.ra_forward_ws(Q, K, V, OUT, LSE, 1, 4, 2, 256, 128, 2, 0, 1, 5, 0, None, 0,
                           None) == rb.RA_ERR_INVALID_ARG


def test_workspace_sizes():
    B, H, Hkv, S, d, N = 1, 4, 2, 512, 128, 4
    # contiguous fused bf16 needs no scratch at all
    assert ra.workspace_bytes(B, H, Hkv, S, d, N, "contiguous", True, "fused") == 0
    striped = ra.workspace_bytes(B, H, Hkv, S, d, N, "striped", True, "fused")
    # q', k', v', out' (bf16) and lse' (fp32), each 256-byte aligned
    assert striped == 2 * (B * H * S * d) * 2 + 2 * (B * Hkv * S * d) * 2 + B * H * S * 4
    per_step = ra.workspace_bytes(B, H, Hkv, S, d, N, "contiguous", True, "per_step")
    assert per_step == 2 * (B * H * S * d * 4 + B * H * S * 4)
    ring = ra.workspace_bytes(B, H, Hkv, S, d, N, "contiguous", True, "ring")
    # plus two rotating copies of k and v (bf16)
    assert ring == per_step + 4 * (B * Hkv * S * d) * 2
    assert ra.workspace_bytes(B, H, Hkv, S, d, 1, "contiguous", True, "ring") == per_step
    assert ra.workspace_bytes(B, 3, 2, S, d, N) == 0  # invalid request -> 0
    assert ra.lib().ra_workspace_bytes(B, H, Hkv, S, d, N, 0, 1, 3, 0) == 0  # unknown mode


def test_permute_and_merge_validation():
    L = ra.lib()
    assert L.ra_permute(Q, K, 1, 1, 30, 8, 2, 4, 0, None) == rb.RA_ERR_INVALID_ARG   # S % N
    assert L.ra_permute(Q, K, 1, 1, 32, 8, 3, 4, 0, None) == rb.RA_ERR_INVALID_ARG   # elem size
    assert L.ra_permute(Q, Q, 1, 1, 32, 8, 2, 4, 0, None) == rb.RA_ERR_INVALID_ARG   # in place
    assert L.ra_merge(Q, K, V, OUT, 10, 6, None) == rb.RA_ERR_INVALID_ARG           # d % 4
    assert L.ra_merge(Q, K, Q, OUT, 10, 8, None) == rb.RA_ERR_INVALID_ARG           # aliasing


def test_every_declared_function_has_ctypes_signature():
    """Sizes above 2^31 (workspaces, row counts) must not be truncated: every
    entry point the header declares gets explicit argument types."""
    L = ra.lib()
    for n in rb.header_functions():
        f = getattr(L, n)
        if n in ("ra_version", "ra_launch_count"):
            continue
        assert f.argtypes is not None, n


def _header_param_counts():
    import re
    with open(rb.HEADER) as fh:
        text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
    counts = {}
    for m in re.finditer(r"\b(ra_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = m.group(2).strip()
        counts[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return counts


def test_ctypes_signatures_match_header_arity():
    """A wrong argument count shifts every later argument; check each binding
    against the number of parameters the header declares."""
    L = ra.lib()
    counts = _header_param_counts()
    assert set(counts) == set(rb.header_functions())
    for n, c in counts.items():
        f = getattr(L, n)
        got = len(f.argtypes) if f.argtypes is not None else 0
        assert got == c, (n, got, c)


def test_ulysses_validation_without_gpu():
    """Requests the library rejects before touching the GPU."""
    L = ra.lib()
    # Hkv = 2 cannot be split over 4 devices
    assert L.ra_ulysses_workspace_bytes(1, 8, 2, 1024, 128, 4, 1, 0) == 0
    assert L.ra_forward_ulysses(Q, K, V, OUT, LSE, 1, 8, 2, 1024, 128, 4, 1, 0, None, 0, None) == \
        rb.RA_ERR_UNSUPPORTED
    # S % n_dev
    assert L.ra_forward_ulysses(Q, K, V, OUT, LSE, 1, 8, 8, 1000, 128, 3, 1, 0, None, 0, None) == \
        rb.RA_ERR_INVALID_ARG
    # a valid request without workspace
    need = L.ra_ulysses_workspace_bytes(1, 8, 4, 1024, 128, 4, 1, 0)
    assert need == 2 * (8 * 1024 * 128 * 2) + 2 * (4 * 1024 * 128 * 2) + 8 * 1024 * 4
    assert L.ra_forward_ulysses(Q, K, V, OUT, LSE, 1, 8, 4, 1024, 128, 4, 1, 0, None, 0, None) == \
        rb.RA_ERR_WORKSPACE
    assert L.ra_all_to_all(Q, K, 1, 6, 32, 8, 2, 4, 0, None) == rb.RA_ERR_INVALID_ARG   # Hn % n


def test_header_is_plain_c_and_a_c_program_links(tmp_path):
    """include/ra.h compiles as C99 (-pedantic, no C++), and a C program that
    includes it links against libra.so and runs the host-only entry points."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    inc = os.path.join(root, "include")
    libdir = os.path.dirname(ra.binding.LIB_PATH)
    src = tmp_path / "use_ra.c"
    src.write_text(
        '#include <stdio.h>\n#include "ra.h"\n'
        "int main(void) {\n"
        "    long long pairs[16], tiles[16];\n"
        "    long long total = ra_schedule_stats(RA_LAYOUT_STRIPED, 1, 4, 256, pairs, tiles);\n"
        '    printf("%s|%s|%lld\\n", ra_version(), ra_status_string(RA_ERR_TIMEOUT), total);\n'
        "    return total > 0 ? 0 : 1;\n"
        "}\n")
    exe = tmp_path / "use_ra"
    res = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, str(src),
                          "-L", libdir, "-lra", "-Wl,-rpath," + libdir, "-o", str(exe)],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stderr
    version, timeout_name, total = run.stdout.strip().split("|")
    assert version == ra.version() and "TIMEOUT" in timeout_name.upper()
    S = 4 * 256
    assert int(total) == S * (S + 1) // 2
