"""The bounds-checking debug build on the parity workloads.

libattn_bwd_gb300_bounds.so is the library compiled with -DFA_DEBUG_BOUNDS: every
TMA tile coordinate, bulk copy range and global store or reduction index is checked
against the extents of its tensor, and a failed check records FA_ERR_BOUNDS and skips
the access.  A child process that loads this build instead of the normal one runs the
forward and the backward (both dQ modes) on shapes that reach every check site --
ragged tails, N = 1, GQA, Nq != Nkv, packed batches with empty sequences, strided
(BSHD) tensors, additive bias with dBias, and the seeded sweep of mixed shapes of
test_random_shapes.py -- and compares every output with the fp64 oracle
(max|err| <= 1e-2 * max|ref| + 1e-3).  The status word must stay FA_OK throughout: on
valid inputs no check fires.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)

CHILD = r"""
import sys
sys.path.insert(0, {tests!r})
sys.path.insert(0, {root!r})
from attn_bwd_gb300 import _lib, inputs
assert _lib.LIB_PATH.endswith("libattn_bwd_gb300_bounds.so"), _lib.LIB_PATH
import test_parity, test_varlen, test_bias, test_strided, test_random_shapes
for shape in test_random_shapes._shapes():
    test_random_shapes.test_random_shape(shape)
for det in (False, True):
    test_parity.check_full(inputs.tiny_mha()[0], 1, det)
    for shape in inputs.ragged():
        test_parity.check_full(shape, 2, det)
    test_parity.check_full(inputs.llama_gqa(256), 5, det)
    test_parity.check_full(inputs.Shape(1, 4, 2, 77, 200, 64, True, "bf16"), 6, det)
    test_parity.check_full(inputs.Shape(2, 6, 3, 129, 257, 128, False, "bf16"), 6, det)
    for pk in inputs.packed_mix()[:4]:
        test_varlen.test_packed_batch(pk, det)
    test_bias.test_bias_broadcast_shapes((2, 4), 1, det)
    test_bias.test_bias_on_packed_batch(2, det)
    test_strided.test_token_major_packed_batch(det)
test_strided.test_bshd_storage_matches_contiguous(96, 1)
assert _lib.fa_last_device_error() == _lib.FA_OK
print("bounds build ok")
"""


def test_bounds_checking_build_matches_the_oracle():
    from attn_bwd_gb300 import build
    lib = build.build(debug_bounds=True)
    code = CHILD.format(tests=TESTS, root=ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=1200,
                       env=dict(os.environ, ATTN_BWD_GB300_LIB=lib))
    assert r.returncode == 0 and "bounds build ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
