"""The C-ABI library builds for sm_103a, loads, and exports every function the
header declares; host-side validation answers without a GPU (no compute calls)."""
import ctypes
import subprocess

import pytest

import oracle
from mixture_experts_expert_gb300 import binding as B
from mixture_experts_expert_gb300 import build as Bld


@pytest.fixture(scope="module")
def lib():
    Bld.build()
    return B.lib()


def test_every_declared_symbol_is_exported(lib):
    names = B.declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/moe_gb300.h but not exported"
    # nothing but the moe_ prefix leaks out of the shared object
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = [line.split()[-1] for line in out.splitlines() if line.strip()]
    assert exported and all(s.startswith("moe_") for s in exported), exported
    assert sorted(exported) == names


def test_host_entry_points_from_plain_c(lib, tmp_path):
    """The header compiles as C99 and the host-only calls work from a C program."""
    import os
    here = os.path.dirname(os.path.abspath(__file__))
    exe = tmp_path / "abi_from_c"
    inc = os.path.join(os.path.dirname(here), "include")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", inc,
                    os.path.join(here, "abi_from_c.c"), B.LIB_PATH,
                    "-Wl,-rpath," + os.path.dirname(B.LIB_PATH), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "FAIL" not in out.stdout and out.stdout.count("ok ") >= 12


def test_library_is_sm103a_only():
    assert "arch=compute_103a,code=sm_103a" in " ".join(Bld.ARCH)


def test_abi_version_and_status_strings(lib):
    assert B.moe_abi_version() == 5
    assert B.moe_status_string(0) == "ok"
    assert "invalid" in B.moe_status_string(-1)
    assert B.moe_status_string(12345) == "unknown status"


@pytest.mark.parametrize("T,K,E,align", [(8192, 8, 128, 128), (256, 2, 8, 128), (5, 3, 7, 16),
                                         (0, 2, 4, 128), (8192, 1, 16, 128)])
def test_capacity_matches_oracle(lib, T, K, E, align):
    assert B.moe_capacity(T, K, E, align) == oracle.capacity(T, K, E, align)


def test_invalid_sizes_rejected_on_host(lib):
    assert B.moe_capacity(8, 0, 4, 128) == 0
    assert B.moe_capacity(8, 2, 0, 128) == 0
    assert B.moe_capacity(8, 2, 2048, 128) == 0
    assert B.moe_workspace_bytes(8, 2, 4, 256, 128, 0) == 0
    L = B.lib()
    # invalid sizes return MOE_ERR_INVALID_ARG before any CUDA call
    nul = ctypes.c_void_p(0)
    st = L.moe_route_permute(nul, nul, nul, 8, 0, 4, 256, 128, nul, nul, nul, nul, nul, nul, nul,
                             nul)
    assert st == B.MOE_ERR_INVALID_ARG
    st = L.moe_combine(nul, nul, nul, 4, 2, 250, nul, nul)   # D not a multiple of 8
    assert st == B.MOE_ERR_INVALID_ARG
    # GEMM shapes the kernels do not tile are reported as unsupported
    st = L.moe_expert_mlp_fwd(nul, nul, nul, nul, nul, nul, 8, 2, 4, 200, 128, 128, nul, nul,
                              nul)
    assert st == B.MOE_ERR_UNSUPPORTED
    st = L.moe_expert_mlp_fwd(nul, nul, nul, nul, nul, nul, 8, 2, 4, 256, 128, 64, nul, nul,
                              nul)
    assert st == B.MOE_ERR_UNSUPPORTED
    st = L.moe_expert_mlp_bwd(nul, nul, nul, nul, nul, nul, nul, nul, nul, nul, 8, 2, 4, 256,
                              96, 128, nul, nul, nul, nul, nul, nul, nul, nul)
    assert st == B.MOE_ERR_UNSUPPORTED
    # null buffers are rejected
    st = L.moe_expert_mlp_fwd(nul, nul, nul, nul, nul, nul, 8, 2, 4, 256, 128, 128, nul, nul,
                              nul)
    assert st == B.MOE_ERR_INVALID_ARG


def test_workspace_grows_with_every_dimension(lib):
    base = B.moe_workspace_bytes(8192, 8, 128, 2048, 768, 128)
    assert base > 0
    cap = oracle.capacity(8192, 8, 128, 128)
    # act [cap,I] + dH [cap,2I] + dy_perm [cap,D] in bf16 at least
    assert base >= cap * (768 * 2 + 768 * 4 + 2048 * 2)
    assert B.moe_workspace_bytes(8192, 8, 128, 4096, 768, 128) > base
    assert B.moe_workspace_bytes(8192, 8, 128, 2048, 1536, 128) > base
    assert B.moe_workspace_bytes(16384, 8, 128, 2048, 768, 128) > base


def test_kernel_names_and_counters(lib):
    names = B.kernel_names()
    assert "gemm_gateup_swiglu" in names and "gemm_dw_down" in names and "combine" in names and "bwd_prep_rows" in names
    total, per = B.moe_launch_count()
    assert total == sum(per.values())
