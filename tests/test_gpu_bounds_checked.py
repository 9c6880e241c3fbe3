"""The parity sweep under the bounds-checked build of the library.

libdcc_checked.so is the same library compiled with DCC_CHECK_BOUNDS=1: every
data access of the collective and fused-layer kernels is checked against the
byte range the call gave its pointer, and the first access outside would be
skipped and reported by dcc_comm_check as DCC_ERR_BOUNDS (with the buffer's
rank, kind and offset).  With compute-sanitizer unavailable this is the
device-side evidence that no kernel reads or writes outside its buffers: the
parity tests run again in a child process with that library loaded, and every
one of them checks dcc_comm_check == DCC_OK after its calls.  No violation is
planted on the GPU.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# the full-size cases run unchecked elsewhere; here the shapes that reach every
# code path (tails, ragged shards, runtime-N instances, launch shapes, bulk and
# LL kernels, entry barrier, host buffers) at sizes the checked build runs quickly
SELECT = ("parity_sweep or random or ragged or special_values or launch_shape or c3_bf16 or "
          "c1_fp32 or entry_barrier_same or empty_inputs or from_host or allgather_bulk or "
          "integer_data or within_bound or random_shapes or reduce_scatter_op_parity or op_with_entry_barrier or "
          "graph_replay or dependent_chain or fused_layer_chain or every_form")


def test_parity_sweep_clean_under_bounds_checked_build():
    from driven_collective_communication_gb300 import build
    build.build()
    build.build(checked=True)
    env = dict(os.environ, DCC_CHECK_BOUNDS="1")
    files = ["tests/test_gpu_collectives.py", "tests/test_gpu_reduce_ops.py", "tests/test_gpu_fused.py",
             "tests/test_gpu_fused_mma.py", "tests/test_gpu_pdl.py"]
    probe = subprocess.run([sys.executable, "-c",
                            "from driven_collective_communication_gb300 import dcc; print(dcc.LIB_PATH)"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip().endswith("libdcc_checked.so"), probe.stdout + probe.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", *files, "-m", "gpu", "-x", "-q", "-k", SELECT,
                        "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail
