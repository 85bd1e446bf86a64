"""The boundary from plain C: tests/c_abi_client.c includes include/tstgemm.h and
links libtstgemm.so with gcc (no Python in the process).  On the CPU its host-only
plan's F(i) and work list match the oracle; on the GPU it runs a GEMM through
cudaMalloc'd buffers and checks small-integer results exactly."""
import glob
import os
import subprocess

import pytest

from oracle import schedule as S
from tile_scheduled_tensor_gb300 import _capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.dirname(_capi.LIB_PATH)


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_client")
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-Wall", "-o", exe, os.path.join(ROOT, "tests", "c_abi_client.c"),
                           "-I", os.path.join(ROOT, "include"), "-L", PKG, "-ltstgemm", f"-Wl,-rpath,{PKG}", "-ldl"])
    return exe


def test_c_client_host_plan_matches_oracle(client):
    M, N, K, kind, G, P = 1000, 700, 64, S.GROUPED_M, 8, 37
    out = subprocess.run([client, "map", str(M), str(N), str(K), str(kind), str(G), str(P)], capture_output=True,
                         text=True, check=True).stdout.split("\n")
    tiles, grid = int(out[0].split()[1]), int(out[0].split()[3])
    Mt, Nt = -(-M // 128), -(-N // 128)
    assert tiles == Mt * Nt and grid == P
    got = [tuple(int(x) for x in line.split()) for line in out[1:1 + tiles]]
    assert got == [S.tile_map(kind, G, Mt, Nt, i) for i in range(tiles)]
    n0 = int(out[1 + tiles].split()[1])
    assert [int(x) for x in out[2 + tiles:2 + tiles + n0]] == [s.tile for s in S.work_items(S.PERSISTENT, 0, P, tiles, 1)]


def _cudart():
    for base in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        found = sorted(glob.glob(os.path.join(base, "lib64", "libcudart.so*")))
        if found:
            return found[0]
    return None


@pytest.mark.gpu
def test_c_client_runs_a_gemm_on_the_gpu(client):
    env = dict(os.environ)
    rt = _cudart()
    if rt:
        env["CUDART_PATH"] = rt
    r = subprocess.run([client, "run", "300", "200", "256"], capture_output=True, text=True, env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0 of 60000" in r.stdout
