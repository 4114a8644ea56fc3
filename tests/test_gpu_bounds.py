"""The parity cases again, on the bounds-checked build of the library (-DCSA_DEBUG_BOUNDS): every
kernel store with a computed index checks it against its buffer's extent and, instead of writing
outside, skips the store and raises bit 8 of the device flag, which the parity tests read back
through csa_device_status.  The cases run in a child process (the library is loaded once per
process) with CSA_LIBRARY_VARIANT=bounds: small odd shapes on both projection paths, chains of
chunks, cache rows, the gate bias, batches beyond one token block, the indexer's quantiser, the
entry point that allocates nothing (its scratch stores checked against the fixed array's
capacity), and the time-out path (a test hook of this build only)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_parity_cases_on_the_bounds_checked_build():
    sys.path.insert(0, ROOT)
    from deepseek_v4_compressed_wkv_gb300 import build as b
    lib = b.build(variant="bounds")
    env = dict(os.environ, CSA_LIBRARY_VARIANT="bounds")
    which = subprocess.run([sys.executable, "-c", "import deepseek_v4_compressed_wkv_gb300 as c; "
                            "c.load_library(build_if_missing=False); print(c.library_path())"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert which.returncode == 0 and which.stdout.strip() == lib, which.stdout + which.stderr
    cases = [os.path.join(HERE, "test_gpu_parity.py") + "::" + t for t in (
        "test_small_prefill_state_and_decode", "test_decode_batch_beyond_one_token_tile",
        "test_errors_are_reported_not_raised_on_the_device", "test_decode_steps_in_a_cuda_graph")]
    cases += [os.path.join(HERE, "test_gpu_chunks.py") + "::" + t for t in (
        "test_prefill_chunks_then_decode", "test_prefill_into_cache_rows", "test_chunk_of_many_sequences_across_waves")]
    cases += [os.path.join(HERE, "test_gpu_gate_bias.py"), os.path.join(HERE, "test_gpu_timeout.py"),
              os.path.join(HERE, "test_zz_no_alloc.py")]
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *cases],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
