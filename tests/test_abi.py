"""The C ABI library without a GPU: it builds, loads, exports every entry point
include/dcc.h declares, and its pure host logic (argument checks that come
before any CUDA call, shard ranges, error names) behaves as documented."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT, gpu_available

HEADER = os.path.join(ROOT, "include", "dcc.h")


@pytest.fixture(scope="module")
def dcc():
    from driven_collective_communication_gb300 import build
    build.build()
    from driven_collective_communication_gb300 import dcc as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(dcc_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("dcc_comm_create", "dcc_comm_destroy", "dcc_register_buffer",
                     "dcc_memory_channel_make", "dcc_allreduce", "dcc_reduce_scatter",
                     "dcc_allgather", "dcc_ring_barrier", "dcc_comm_check", "dcc_error_string"):
        assert required in names
    assert len(names) >= 20


def test_library_exports_every_declared_symbol(dcc):
    out = subprocess.run(["nm", "-D", "--defined-only", dcc.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (dcc_\w+)$", out, flags=re.M))
    missing = [f for f in declared_functions() if f not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(dcc.LIB_PATH)
    for f in declared_functions():
        assert getattr(lib, f) is not None


def test_every_exported_symbol_is_declared(dcc):
    """The boundary is exactly the header: no dcc_* entry point is exported
    without a declaration (and its documentation) in include/dcc.h."""
    out = subprocess.run(["nm", "-D", "--defined-only", dcc.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (dcc_\w+)$", out, flags=re.M))
    assert exported <= set(declared_functions()), sorted(exported - set(declared_functions()))


def test_bounds_checked_build_compiles_and_exports_the_same_boundary(dcc):
    """The DCC_CHECK_BOUNDS=1 build of the same sources (libdcc_checked.so)
    compiles and exports exactly the entry points of the default library."""
    from driven_collective_communication_gb300 import build
    path = build.build(checked=True)

    def exported(lib):
        out = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True, text=True,
                             check=True).stdout
        return set(re.findall(r"\bT (dcc_\w+)$", out, flags=re.M))
    assert exported(path) == exported(dcc.LIB_PATH)


def test_build_targets_sm103a_only():
    """The build generates device code for sm_103a alone (one -gencode, no PTX
    for other architectures); the GPU test below checks what the runtime sees."""
    from driven_collective_communication_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert not any("-gencode" in f or "-arch" in f for f in build.NVCC_FLAGS)


@pytest.mark.gpu
def test_every_kernel_runs_as_sm103a_binary(dcc):
    """The CUDA runtime reports binaryVersion 103 for every kernel of the library."""
    import torch
    torch.cuda.set_device(0)
    assert dcc.dcc_kernel_binary_version() == 103


def test_error_strings(dcc):
    for code, name in [(0, "DCC_OK"), (-1, "DCC_ERR_INVALID_ARG"), (-2, "DCC_ERR_NOT_REGISTERED"),
                       (-3, "DCC_ERR_MISALIGNED"), (-4, "DCC_ERR_NO_CHANNEL"), (-5, "DCC_ERR_CUDA"),
                       (-6, "DCC_ERR_LAUNCH"), (-7, "DCC_ERR_TIMEOUT"), (-8, "DCC_ERR_UNSUPPORTED"),
                       (-9, "DCC_ERR_BOUNDS")]:
        assert dcc.dcc_error_string(code) == name
    assert dcc.dcc_error_string(-99) == "DCC_ERR_UNKNOWN"
    assert "sm_103a" in dcc.dcc_version()


def test_create_rejects_bad_rank_counts_before_touching_cuda(dcc):
    h = ctypes.c_void_p()
    for n in (0, -1, 17, 1000):
        assert dcc.raw_call("dcc_comm_create", n, ctypes.byref(h)) == dcc.DCC_ERR_INVALID_ARG
    assert dcc.raw_call("dcc_comm_create", 2, None) == dcc.DCC_ERR_INVALID_ARG


@pytest.mark.skipif(gpu_available(), reason="checks the no-device path")
def test_create_without_device_reports_cuda_error(dcc):
    h = ctypes.c_void_p()
    assert dcc.raw_call("dcc_comm_create", 2, ctypes.byref(h)) == dcc.DCC_ERR_CUDA
    assert not h.value


def test_null_communicator_is_rejected(dcc):
    P = ctypes.POINTER(ctypes.c_void_p)
    arr = (ctypes.c_void_p * 2)()
    i = ctypes.c_int()
    calls = [
        ("dcc_register_buffer", None, 0, 0, ctypes.c_void_p(16), 16),
        ("dcc_memory_channel_make", None, 0, 1),
        ("dcc_allreduce", None, arr, arr, 4, 1, 0, None),
        ("dcc_reduce_scatter", None, arr, arr, 4, 1, None),
        ("dcc_allgather", None, arr, arr, 4, 1, None),
        ("dcc_allreduce_op", None, arr, arr, 4, 1, 1, 0, None),
        ("dcc_reduce_scatter_op", None, arr, arr, 4, 1, 1, None),
        ("dcc_linear_allreduce", None, arr, arr, arr, 8, 8, 3, None),
        ("dcc_linear_allreduce_residual", None, arr, arr, arr, arr, 8, 8, 3, None),
        ("dcc_linear_allreduce_tokens", None, arr, arr, arr, 1, 8, 64, 3, None),
        ("dcc_linear_allreduce_tokens_residual", None, arr, arr, arr, arr, 1, 8, 64, 3, None),
        ("dcc_allreduce_from_host", None, arr, arr, arr, arr, 4, 1, 0, None),
        ("dcc_ring_barrier", None, 1, None),
        ("dcc_comm_check", None, None),
        ("dcc_comm_error_detail", None, None, None, None),
        ("dcc_channel_put", None, 0, 1, 0, 0, 16, 0, None),
        ("dcc_channel_get", None, 0, 1, 0, 0, 16, None),
        ("dcc_comm_read_semaphores", None, 0, None, None, None),
        ("dcc_set_wait_timeout_us", None, 10),
        ("dcc_set_blocks_per_rank", None, 1),
        ("dcc_set_algo_threshold", None, 1, 1024),
        ("dcc_set_entry_barrier", None, 1),
        ("dcc_set_pdl", None, 1),
        ("dcc_select_algo", None, 4, 1, ctypes.byref(i)),
        ("dcc_debug_skip_signal", None, 0),
        ("dcc_launch_shape", None, 4, 1, 0, ctypes.byref(i), ctypes.byref(i)),
        ("dcc_proxy_start", None),
        ("dcc_proxy_stop", None),
        ("dcc_proxy_set_handler", None, None, None),
        ("dcc_proxy_stats", None, None, None),
        ("dcc_port_put", None, 0, 1, 0, 0, 16, 0, 0, None),
        ("dcc_port_allgather", None, arr, arr, 4, 1, None),
        ("dcc_fifo_push", None, None, None, 1, None),
    ]
    for name, *args in calls:
        assert dcc.raw_call(name, *args) == dcc.DCC_ERR_INVALID_ARG, name
    assert dcc.raw_call("dcc_comm_destroy", None) == dcc.DCC_OK


@pytest.mark.parametrize("eb", [2, 4])
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 16])
@pytest.mark.parametrize("count", [0, 1, 7, 8, 63, 64, 1000, 4096 + 5, 33554432])
def test_shard_ranges_partition_the_buffer(dcc, n, count, eb):
    """Two-shot shards are disjoint, cover [0, count), start on 16-byte
    boundaries, and only the last rank holds a partial vector."""
    vw = 16 // eb
    prev_end = 0
    for r in range(n):
        b, e = dcc.dcc_shard_range(count, n, r, eb)
        assert b == prev_end and b <= e
        assert b % vw == 0
        if r < n - 1:
            assert e % vw == 0
        prev_end = e
    assert prev_end == count
    if count >= n * vw:
        sizes = [dcc.dcc_shard_range(count, n, r, eb) for r in range(n)]
        sizes = [e - b for b, e in sizes]
        assert max(sizes[:-1]) == min(sizes[:-1]) if n > 1 else True
        assert sizes[-1] - sizes[0] < n * vw


def test_shard_range_rejects_bad_arguments(dcc):
    b, e = ctypes.c_size_t(), ctypes.c_size_t()
    for args in [(10, 0, 0, 2), (10, 2, 2, 2), (10, 2, -1, 2), (10, 17, 0, 2), (10, 2, 0, 3)]:
        assert dcc.raw_call("dcc_shard_range", *args, ctypes.byref(b), ctypes.byref(e)) == \
            dcc.DCC_ERR_INVALID_ARG


def test_compiled_auto_table_is_the_tuning_json(dcc):
    """AUTO's one-shot thresholds come from one source: the JSON table the
    crossover sweep writes; the library's compiled defaults equal it for every
    rank count and dtype."""
    from driven_collective_communication_gb300 import build
    table = build.load_auto_table()
    for n in range(1, 17):
        for t in ("int32", "fp32", "fp16", "bf16"):
            assert dcc.dcc_auto_threshold(n, t) == table[n][t], (n, t)
    for bad in ((0, "bf16"), (17, "bf16")):
        with pytest.raises(dcc.DccError):
            dcc.dcc_auto_threshold(*bad)


def test_python_binding_names_match_the_header(dcc):
    """The binding wraps each C entry point under the same name."""
    for f in declared_functions():
        assert hasattr(dcc, f), f


def test_product_path_does_not_touch_the_oracle():
    """Nothing under the package (binding, build, kernels) imports, loads or
    includes anything of the oracle."""
    pkg = os.path.join(ROOT, "driven_collective_communication_gb300")
    pat = re.compile(r"(^\s*(import|from)\s+oracle\b|liboracle|oracle\.c\b|oracle/)", re.M)
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, fn)).read()
                assert not pat.search(text), os.path.join(dirpath, fn)


def test_c_example_compiles_and_links(dcc, tmp_path):
    """The C caller under examples/ compiles against include/dcc.h and links
    against libdcc.so (every dcc_* call it makes resolves)."""
    src = os.path.join(ROOT, "driven_collective_communication_gb300", "examples", "allreduce_8_ranks.c")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    obj = tmp_path / "example.o"
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-I", os.path.join(cuda, "include"), "-c", src, "-o", str(obj)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    main = tmp_path / "main.c"
    main.write_text("int main(void) { return 0; }\n")
    libdir = os.path.dirname(dcc.LIB_PATH)
    cudalib = os.path.join(cuda, "lib64")
    r = subprocess.run(["gcc", str(main), str(obj), "-L", libdir, "-ldcc", "-L", cudalib, "-lcudart",
                        "-Wl,-rpath-link," + cudalib, "-o", str(tmp_path / "example")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
