"""The C-ABI library builds, loads and exports every symbol include/*.h declares;
its host-only planner matches the oracle (CPU only, no CUDA calls)."""
import glob
import os
import re
import subprocess

import pytest

from synth import shapes

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from ring_all_reduce_ddp_gb300 import build
    build.build_library()
    import ring_all_reduce_ddp_gb300 as d
    return d


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(ddp_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(L):
    declared = _declared()
    assert declared, "no declarations found"
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (ddp_\w+)", out))
    assert declared <= exported, declared - exported
    # and nothing else: no C++ internals or template instances leak out
    every = set(line.split()[-1] for line in out.splitlines() if line.strip())
    assert every == exported == declared, sorted(every - declared)[:10]
    # and the binding knows every one of them, under the same name
    assert declared <= set(L.exported_symbols())
    for name in declared:
        assert hasattr(L.lib(), name)


def test_status_strings(L):
    assert L.status_string(L.DDP_OK) == "DDP_OK"
    assert L.status_string(L.DDP_ERR_NOT_DIVISIBLE) == "DDP_ERR_NOT_DIVISIBLE"


@pytest.mark.parametrize("builder,esize", [(shapes.tiny, 4), (shapes.resnet50, 4), (shapes.gpt2_small, 4),
                                            (shapes.llama_1b, 2)])
@pytest.mark.parametrize("order", ["reversed", "registration"])
def test_bucket_assign_matches_oracle(L, builder, esize, order):
    from oracle import buckets as ob
    numel = [shapes.numel(s) for _, s in builder()]
    first, cap = ((16 << 10), (256 << 10)) if builder is shapes.tiny else ((1 << 20), (25 << 20))
    want = ob.assign_buckets(numel, esize, first, cap, order)
    _, off, bn = ob.bucket_layout(numel, want)
    got = L.ddp_bucket_assign(numel, esize, first, cap,
                              L.DDP_ORDER_REVERSED if order == "reversed" else L.DDP_ORDER_REGISTRATION)
    assert got["buckets"] == want
    assert got["offset"] == off and got["bucket_numel"] == bn


@pytest.mark.parametrize("seed", range(30))
def test_bucket_assign_random_edge_cases(L, seed):
    import numpy as np
    from oracle import buckets as ob
    rng = np.random.default_rng(seed)
    k = int(rng.integers(0, 20))
    numel = [int(x) for x in rng.integers(0, 50, size=k)]
    first, cap = int(rng.integers(0, 100)), int(rng.integers(0, 300))
    for order, code in (("reversed", L.DDP_ORDER_REVERSED), ("registration", L.DDP_ORDER_REGISTRATION)):
        assert L.ddp_bucket_assign(numel, 4, first, cap, code)["buckets"] == \
            ob.assign_buckets(numel, 4, first, cap, order)


def test_argument_errors_are_reported_before_any_launch(L):
    with pytest.raises(L.DDPError) as e:
        L.ddp_bucket_assign([1, -2], 4, 16, 16)
    assert e.value.status == L.DDP_ERR_ARG
    lib = L.lib()
    import ctypes
    arr = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    assert lib.ddp_allreduce(arr, 0, 10, 0, 1.0, 0, None) == L.DDP_ERR_ARG          # p = 0
    assert lib.ddp_allreduce(arr, 2, 10, 7, 1.0, 0, None) == L.DDP_ERR_DTYPE        # bad dtype
    assert lib.ddp_allreduce(arr, 2, 10, 0, 0.0, 0, None) == L.DDP_ERR_ARG          # divisor 0
    assert lib.ddp_allreduce(arr, 2, 2000, 0, 1.0, 0, None) == L.DDP_ERR_ARG        # overlap
    assert "overlap" in L.ddp_last_error()
    assert lib.ddp_reduce_scatter(arr, (ctypes.c_void_p * 2)(0x10000, 0x20000), 2, 11, 0, 1.0,
                                  L.DDP_OWN_RANK, 0, None) == L.DDP_ERR_NOT_DIVISIBLE
    assert lib.ddp_broadcast(arr, 2, 16, 5, 0, None) == L.DDP_ERR_ARG                # root out of range
    # zero-size work is a no-op that touches no device
    assert lib.ddp_allreduce(arr, 2, 0, 0, 1.0, 0, None) == L.DDP_OK
    assert lib.ddp_reducer_num_buckets(None) == -1 and lib.ddp_reducer_staged(None) == -1


@pytest.mark.parametrize("seed", range(20))
def test_bucket_assign_order_matches_oracle_rebuild(L, seed):
    import numpy as np
    from oracle import reducer_sim as rs
    rng = np.random.default_rng(seed)
    k = int(rng.integers(1, 40))
    numel = [int(x) for x in rng.integers(0, 5000, size=k)]
    walk = [int(x) for x in rng.permutation(k)]
    first, cap = int(rng.integers(0, 20000)), int(rng.integers(1, 60000))
    got = L.ddp_bucket_assign_order(numel, 4, first, cap, walk)
    assert got["buckets"] == rs.rebuild(numel, 4, first, cap, walk)
    with pytest.raises(L.DDPError):
        L.ddp_bucket_assign_order(numel, 4, first, cap, walk[:-1] + [walk[0]] if k > 1 else [5])


def test_missing_library_fails_loudly(tmp_path):
    """With the shared object absent the binding raises on first use: there is
    no CPU or PyTorch fallback anywhere on the product path."""
    import subprocess
    import sys
    code = (
        "import ring_all_reduce_ddp_gb300 as D\n"
        f"D.LIB_PATH = {str(tmp_path / 'absent.so')!r}\n"
        "try:\n"
        "    D.ddp_allreduce([0, 0], 0, D.DDP_FLOAT32, 2.0, stream=0)\n"
        "except RuntimeError as e:\n"
        "    assert 'not built' in str(e), e\n"
        "    print('raised')\n"
    )
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120,
                       env=dict(os.environ, PYTHONPATH=ROOT))
    assert r.returncode == 0 and r.stdout.strip() == "raised", r.stderr


def test_binding_rejects_tensors_it_cannot_pass_as_pointers(L):
    """The library sees a first byte and an element count: the binding refuses
    host tensors, non-contiguous views, and a Reducer whose replicas disagree
    on sizes or mix dtypes, before anything reaches the library."""
    torch = pytest.importorskip("torch")
    host = [torch.zeros(8) for _ in range(2)]
    with pytest.raises(ValueError, match="CUDA device"):
        L.ddp_allreduce(host, 8, L.DDP_FLOAT32, 2.0, stream=0)
    mixed = [[torch.zeros(4), torch.zeros(4, dtype=torch.bfloat16)] for _ in range(2)]
    with pytest.raises(ValueError, match="one dtype"):
        L.DDPReducer(mixed)
    ragged = [[torch.zeros(4)], [torch.zeros(5)]]
    with pytest.raises(ValueError, match="sizes"):
        L.DDPReducer(ragged)


@pytest.mark.gpu
def test_binding_rejects_non_contiguous_views(L):
    torch = pytest.importorskip("torch")
    bufs = [torch.zeros(16, device="cuda")[::2] for _ in range(2)]
    with pytest.raises(ValueError, match="contiguous"):
        L.ddp_allreduce(bufs, 8, L.DDP_FLOAT32, 2.0)


def test_c_program_compiles_against_the_header_alone(L, tmp_path):
    """The header is enough to build a C++ user of the library (no torch, no
    Python): tests/c/abi_smoke.cpp compiles and links here; the GPU tests run it."""
    from ring_all_reduce_ddp_gb300 import build as B
    lib = B.build_library()
    cmd = [B.nvcc(), *B.ARCH, "-O2", "-std=c++17", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_smoke.cpp"), "-L", os.path.dirname(lib), "-lddp_ring",
           "-o", str(tmp_path / "abi_smoke")]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]


def test_header_compiles_as_plain_c(tmp_path):
    """include/ddp_ring.h is a C header: it compiles as C99 (only the CUDA
    runtime's stream type is needed from outside)."""
    import shutil
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if gcc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are not available")
    src = tmp_path / "use_header.c"
    src.write_text('#include "ddp_ring.h"\nint main(void) { return ddp_reducer_staged(0) == -1 ? 0 : 1; }\n')
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
                        "-I", cuda_inc, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
