"""Randomized parity sweep through the C ABI: seeded draws of the layout, the
shape (ragged in every dimension), the FP8 format of B, the output type and
the tile plan (forced through the process-wide knobs: tile width, split-K
cluster size, CTA pairs, the store warp, swapped operand roles), each call
compared element by element with the CPU oracle.  Grouped calls start from a
sentinel-filled D, and the rows they must leave untouched are checked bit for
bit.  The hand-picked cases of the other GPU tests pin each feature; this
sweep covers their combinations."""
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from random_cases import random_case, reset_knobs  # noqa: E402

N_CASES = 160


@pytest.fixture
def knobs():
    yield
    reset_knobs()


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_call_matches_oracle(knobs, case):
    if not random_case(case, rng_base=20_000, seed_base=0):
        pytest.skip("no rows drawn")
