"""The C ABI library builds, loads and exports every entry point that include/dg.h declares; argument
checks that need no GPU reject bad calls before any CUDA work (CPU only)."""
import ctypes
import json
import os
import re

import pytest

import moe_grouped_gemm_tma_gb300 as dg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


def declared_symbols():
    syms = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            text = open(os.path.join(INCLUDE, h)).read()
            syms.update(re.findall(r"^\s*(?:dg_status|const char\*|int|void)\s+(dg_\w+)\s*\(", text, flags=re.M))
    return sorted(syms)


def test_header_declares_every_operation():
    syms = declared_symbols()
    for s in ("dg_gemm_fp8_nt", "dg_m_grouped_contiguous", "dg_m_grouped_masked", "dg_k_grouped_wgrad",
              "dg_wgrad_fp8_nt", "dg_gemm_fp8", "dg_gemm_fp8_nt_ue8m0", "dg_gemm_fp8_nt_ue8m0_packed",
              "dg_status_string", "dg_device_status"):
        assert s in syms


def test_library_exports_every_declared_symbol():
    L = dg.load()
    for s in declared_symbols():
        assert hasattr(L, s), s


def test_python_binding_has_the_same_names():
    for s in declared_symbols():
        assert callable(getattr(dg, s)), s


def test_tuning_knobs_set_get_and_reset():
    dg.dg_tuning_reset()
    assert all(dg.dg_tuning_get(k) == -1 for k in dg.TUNE_KNOBS)
    with dg.tuning(bn=128, split=4):
        assert dg.dg_tuning_get("bn") == 128 and dg.dg_tuning_get("split") == 4
        assert dg.dg_tuning_get("pair") == -1
    assert dg.dg_tuning_get("bn") == -1 and dg.dg_tuning_get("split") == -1
    with pytest.raises(dg.DGError):
        dg.dg_tuning_set(99, 1)
    assert dg.load().dg_tuning_get(99) == -1


def test_environment_is_read_only_with_the_opt_in():
    # a stray DG_* variable must not change the product path; DG_TUNING=1 makes the library read them
    # once, at load
    import subprocess
    import sys
    code = ("import moe_grouped_gemm_tma_gb300 as dg; "
            "print(dg.dg_tuning_get('bn'), dg.dg_tuning_get('split'), dg.dg_tuning_get('pdl'))")
    env = dict(os.environ, DG_BN="64", DG_SPLIT="2", DG_PDL="0")
    env.pop("DG_TUNING", None)
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, check=True)
    assert out.stdout.split() == ["-1", "-1", "-1"]
    env["DG_TUNING"] = "1"
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, check=True)
    assert out.stdout.split() == ["64", "2", "0"]


def test_wait_timeout_hook_rejects_a_zero_limit():
    assert dg.load().dg_testing_arm_wait_timeout(0) == 1          # DG_INVALID_ARG, nothing armed


def test_status_strings():
    assert dg.dg_status_string(0) == "DG_OK"
    assert dg.dg_status_string(6) == "DG_DEVICE_TIMEOUT"
    assert dg.dg_status_string(99) == "DG_UNKNOWN_STATUS"


def _fake(addr):
    return ctypes.c_void_p(addr)


def test_rejects_bad_shapes_before_any_cuda_call():
    L = dg.load()
    ok = _fake(0x10000)
    assert L.dg_gemm_fp8_nt(ok, ok, ok, ok, ok, -1, 8, 128, None) == 1
    assert L.dg_gemm_fp8_nt(ok, ok, ok, ok, ok, 0, 8, 128, None) == 0          # empty: no-op
    assert L.dg_gemm_fp8_nt(ok, ok, ok, ok, ok, 4, 8, 100, None) == 2          # K % 128
    assert L.dg_gemm_fp8_nt(ok, ok, ok, ok, ok, 4, 12, 128, None) == 2         # N % 8
    assert L.dg_gemm_fp8_nt(ok, ok, ok, ok, _fake(0x10008), 4, 8, 128, None) == 3  # D misaligned
    assert L.dg_gemm_fp8_nt(ok, ok, ok, ok, None, 4, 8, 128, None) == 1
    assert L.dg_gemm_fp8(ok, ok, ok, ok, ok, 24, 16, 128, 1, 0, None) == 2     # A stored [K, M], M % 16
    assert L.dg_gemm_fp8(ok, ok, ok, ok, ok, 16, 24, 128, 0, 1, None) == 2     # B stored [K, N], N % 16
    assert L.dg_gemm_fp8(ok, ok, ok, ok, ok, 0, 16, 128, 1, 1, None) == 0      # empty: no-op
    assert L.dg_m_grouped_contiguous(ok, ok, ok, ok, ok, ok, 100, 8, 128, 2, None) == 2  # Mt % 128
    assert L.dg_m_grouped_contiguous(ok, ok, ok, ok, ok, ok, 128, 8, 128, 0, None) == 1  # G = 0
    assert L.dg_m_grouped_masked(ok, ok, ok, ok, ok, ok, 2000, 64, 8, 128, 0, None) == 1  # G too large
    assert L.dg_m_grouped_masked(ok, ok, ok, ok, ok, ok, 2, 64, 8, 130, 0, None) == 2
    ks = (ctypes.c_int32 * 2)(128, 100)
    assert L.dg_k_grouped_wgrad(ok, ok, ok, ok, ks, ok, 2, 8, 8, None) == 2   # ks % 128
    ks = (ctypes.c_int32 * 2)(128, -128)
    assert L.dg_k_grouped_wgrad(ok, ok, ok, ok, ks, ok, 2, 8, 8, None) == 1
    ks = (ctypes.c_int32 * 2)(0, 0)
    assert L.dg_k_grouped_wgrad(ok, ok, ok, ok, ks, ok, 2, 8, 8, None) == 0   # nothing to add
    assert L.dg_wgrad_fp8_nt(ok, ok, ok, ok, ok, 8, 8, 100, 1, None) == 2        # K % 128
    assert L.dg_wgrad_fp8_nt(ok, ok, ok, ok, ok, 8, 12, 128, 1, None) == 2       # N % 8
    assert L.dg_wgrad_fp8_nt(ok, ok, ok, ok, ok, -1, 8, 128, 1, None) == 1
    assert L.dg_wgrad_fp8_nt(ok, ok, ok, ok, ok, 8, 8, 0, 1, None) == 0          # K = 0, accumulate: no-op
    assert L.dg_wgrad_fp8_nt(ok, ok, ok, ok, _fake(0x10008), 8, 8, 0, 0, None) == 3  # zeroing misaligned D
    for f in (L.dg_gemm_fp8_nt_ue8m0, L.dg_gemm_fp8_nt_ue8m0_packed):
        assert f(ok, ok, ok, ok, ok, -1, 8, 128, None) == 1
        assert f(ok, ok, ok, ok, ok, 0, 8, 128, None) == 0                       # empty: no-op
        assert f(ok, ok, ok, ok, ok, 4, 8, 100, None) == 2                       # K % 128
        assert f(ok, ok, ok, ok, ok, 4, 12, 128, None) == 2                      # N % 8
        assert f(ok, ok, ok, ok, _fake(0x10008), 4, 8, 128, None) == 3           # D misaligned
        assert f(ok, ok, ok, ok, None, 4, 8, 128, None) == 1


def test_scale_shapes_follow_the_pages_usage_example():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "page_usage_example.json")))
    sfa, sfb = dg.scale_shapes(g["M"], g["N"], g["K"])
    assert list(sfa) == g["sfa_shape"] and list(sfb) == g["sfb_shape"]


def test_grouped_entry_points_check_arguments_before_any_cuda_call():
    L = dg.load()
    ok, odd16, odd4 = _fake(0x10000), _fake(0x10008), _fake(0x10002)
    # contiguous: (A, sfa, B, sfb, m_indices, D, Mt, N, K, G)
    C = L.dg_m_grouped_contiguous
    assert C(ok, ok, ok, ok, ok, ok, 0, 8, 128, 2, None) == 0           # no rows: no-op
    assert C(ok, ok, ok, ok, ok, ok, 128, 0, 128, 2, None) == 0         # no columns: no-op
    assert C(ok, ok, ok, ok, ok, ok, 128, 8, 128, -1, None) == 1
    assert C(ok, ok, ok, ok, ok, ok, 128, 8, 0, 2, None) == 2           # K = 0 has no expert product
    assert C(ok, ok, ok, ok, ok, ok, 128, 12, 128, 2, None) == 2        # N % 8
    assert C(ok, ok, ok, ok, None, ok, 128, 8, 128, 2, None) == 1       # no m_indices
    assert C(odd16, ok, ok, ok, ok, ok, 128, 8, 128, 2, None) == 3      # A not 16-byte aligned
    assert C(ok, odd4, ok, ok, ok, ok, 128, 8, 128, 2, None) == 3       # sfa not 4-byte aligned
    assert C(ok, ok, ok, ok, odd4, ok, 128, 8, 128, 2, None) == 3       # m_indices not 4-byte aligned
    # masked: (A, sfa, B, sfb, masked_m, D, G, max_m, N, K, expected_m)
    Mk = L.dg_m_grouped_masked
    assert Mk(ok, ok, ok, ok, ok, ok, 0, 64, 8, 128, 0, None) == 0      # no experts: no-op
    assert Mk(ok, ok, ok, ok, ok, ok, 2, 0, 8, 128, 0, None) == 0       # no rows: no-op
    assert Mk(ok, ok, ok, ok, ok, ok, 2, -1, 8, 128, 0, None) == 1
    assert Mk(ok, ok, ok, ok, ok, ok, 1025, 64, 8, 128, 0, None) == 1   # above the 1024-expert limit
    assert Mk(ok, ok, ok, ok, ok, ok, 2, 64, 8, 0, 0, None) == 2
    assert Mk(ok, ok, ok, ok, ok, ok, 2, 64, 12, 128, 0, None) == 2
    assert Mk(ok, ok, ok, ok, None, ok, 2, 64, 8, 128, 0, None) == 1    # no masked_m
    assert Mk(ok, ok, ok, ok, ok, odd16, 2, 64, 8, 128, 0, None) == 3   # D not 16-byte aligned
    assert Mk(ok, ok, ok, ok, odd4, ok, 2, 64, 8, 128, 0, None) == 3    # masked_m not 4-byte aligned
    assert Mk(ok, ok, ok, ok, ok, ok, 2, 1 << 30, 8, 128, 0, None) == 2  # G * max_m rows beyond int32
    # k-grouped: (A, sfa, B, sfb, ks_host, D, G, M, N)
    K = L.dg_k_grouped_wgrad
    ks2 = (ctypes.c_int32 * 2)(128, 256)
    assert K(ok, ok, ok, ok, ks2, ok, 2, 0, 8, None) == 0               # no rows: no-op
    assert K(ok, ok, ok, ok, ks2, ok, -1, 8, 8, None) == 1
    assert K(ok, ok, ok, ok, None, ok, 2, 8, 8, None) == 1              # no ks
    assert K(ok, ok, ok, ok, (ctypes.c_int32 * 129)(*([128] * 129)), ok, 129, 8, 8, None) == 1  # above 128 experts
    assert K(ok, ok, ok, ok, ks2, ok, 2, 8, 12, None) == 2              # N % 8
    assert K(None, ok, ok, ok, ks2, ok, 2, 8, 8, None) == 1             # no A
    assert K(ok, ok, ok, odd4, ks2, ok, 2, 8, 8, None) == 3             # sfb not 4-byte aligned
    assert K(ok, ok, ok, ok, ks2, odd16, 2, 8, 8, None) == 3            # D not 16-byte aligned
    big = (ctypes.c_int32 * 2)((1 << 31) - 128, (1 << 31) - 128)
    assert K(ok, ok, ok, ok, big, ok, 2, 8, 8, None) == 2               # sum of ks beyond int32
    assert K(ok, ok, ok, ok, ks2, ok, 2, 1 << 30, 8, None) == 2         # G * M beyond int32


def test_binding_has_no_cpu_path():
    # host tensors are refused before the library is called: there is no CPU fallback
    import torch
    from moe_grouped_gemm_tma_gb300 import inputs as I
    c = I.make_normal(I.seed_for(0), 128, 256, 512)
    D = torch.empty(128, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dg.dg_gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb, D)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dg.dg_gemm_fp8_nt_ue8m0(c.A, c.sfa, c.B, c.sfb, D)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dg.dg_wgrad_fp8_nt(c.A, c.sfa, c.A, c.sfa, torch.zeros(128, 128))
    with pytest.raises(TypeError, match="e4m3 codes"):
        dg.dg_gemm_fp8_nt(c.A.float(), c.sfa, c.B, c.sfb, D)


def test_package_never_imports_the_oracle():
    # the product path (binding, build, input generators) does not reach the test oracle
    pkg = os.path.join(ROOT, "moe_grouped_gemm_tma_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", text, flags=re.M), f
                assert "liboracle" not in text and "oracle.cpp" not in text, f


def test_sources_name_no_batched_copy_call():
    # batched host<->device copy calls are closed for this library: every copy is one plain async copy
    # (the pattern is assembled from parts so that this file does not name them either)
    pat = re.compile("(cuda|cu)Memcpy(3D)?" + "Batch" + "Async")
    for dirpath, dirs, files in os.walk(ROOT):
        dirs[:] = [d for d in dirs if d not in (".git", "_work", "gpurun_out", "_build", "__pycache__")]
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp", ".c", ".sh")):
                text = open(os.path.join(dirpath, f), encoding="utf-8", errors="replace").read()
                assert not pat.search(text), os.path.join(dirpath, f)


def test_kernels_report_failures_without_trapping():
    # a kernel that gives up records a status word and returns: no trap and no device-side assert
    csrc = os.path.join(ROOT, "moe_grouped_gemm_tma_gb300", "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f), encoding="utf-8").read()
        assert "__trap" not in text and not re.search(r"\btrap\s*;", text), f
        assert not re.search(r"(?<!static_)\bassert\s*\(", text), f


def test_every_device_loop_without_a_counted_bound_is_a_known_bounded_one():
    # Waits in the kernels end: wait_bounded gives up after a time limit and raises the abort flag (its
    # suspended try_wait returns after at most its hint), drain_wait gives up after a shorter one; the only other open loops are the masked layout's binary
    # search (hi - lo halves each pass) and the host-side stage count. A new open loop must be added
    # here deliberately, with its bound.
    known = {
        "while (s > 1 && 1024 + ((s * stage_bytes + scale_bytes + 1023) / 1024) * 1024 + store_bytes + static_bytes > SMEM_LIMIT)",
        "while (hi - lo > 1) {",
        "while (true) {",                              # wait_bounded: exit on success, abort or time limit
        "while (!mbar_try_wait(bar, parity))",         # drain_wait: exits on success or time limit
    }
    csrc = os.path.join(ROOT, "moe_grouped_gemm_tma_gb300", "csrc")
    found = []
    for f in sorted(os.listdir(csrc)):
        for line in open(os.path.join(csrc, f), encoding="utf-8"):
            code = line.split("//")[0].strip()
            if re.search(r"\bwhile\s*\(|\bfor\s*\(\s*;\s*;", code):
                found.append((f, code))
    assert found, "no loops found: the scan is broken"
    for f, code in found:
        assert code in known, (f, code)
    text = open(os.path.join(csrc, "dg_kernel.cuh"), encoding="utf-8").read()
    body = text[text.index("bool wait_bounded("):text.index("void drain_wait(")]
    assert "WAIT_LIMIT_NS" in body and "abort_flag" in body and "STATUS_TIMEOUT" in body
    # every suspended try_wait carries a finite hint (nanoseconds, an integer literal)
    hints = re.findall(r"mbar_try_wait_hint\([^;]*?,\s*(\d+)\)", "".join(
        open(os.path.join(csrc, f), encoding="utf-8").read() for f in sorted(os.listdir(csrc))))
    assert hints and all(0 < int(h) <= 1_000_000 for h in hints), hints
    body = text[text.index("void drain_wait("):]
    assert "DRAIN_LIMIT_NS" in body[:400]
