"""Each planted mistake in the oracle must make at least one pin fail.

The mistakes are planted in the oracle itself, on the CPU, through
``oracle.set_mutation``; the pins are the functions of ``test_oracle_pins``.
"""
import pytest

import oracle
from tests import test_oracle_pins as pins

MUTANTS = {
    "reversed_ring": oracle.MUT_REVERSED_RING,
    "start_at_owner": oracle.MUT_START_AT_OWNER,
    "drop_scale": oracle.MUT_DROP_SCALE,
    "truncate_cast": oracle.MUT_TRUNCATE_CAST,
    "skip_last_step": oracle.MUT_SKIP_LAST_STEP,
    "gemm_transpose": oracle.MUT_GEMM_TRANSPOSE,
    "pad_not_zero": oracle.MUT_PAD_NOT_ZERO,
    "psum_skip_rank": oracle.MUT_PSUM_SKIP_RANK,
    "odc_settle_per_microbatch": oracle.MUT_ODC_SETTLE_PER_MB,
    "odc_flat_fold": oracle.MUT_ODC_FLAT_FOLD,
    "odc_reversed_microbatches": oracle.MUT_ODC_REVERSED_MB,
    "odc_pairwise_microbatches": oracle.MUT_ODC_PAIRWISE_MB,
    "pipeline_carry_in_fold": oracle.MUT_PIPE_CARRY_IN_FOLD,
    "pipeline_reversed_groups": oracle.MUT_PIPE_REVERSED_GROUPS,
    "pipeline_scale_per_group": oracle.MUT_PIPE_SCALE_PER_GROUP,
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    caught = []
    old = oracle.set_mutation(MUTANTS[name])
    try:
        for pin in pins.PINS:
            try:
                pin()
            except (AssertionError, oracle.OracleError, ValueError):
                caught.append(pin.__name__)
    finally:
        oracle.set_mutation(old)
    assert caught, f"no pin catches the {name} mutation"


def test_unmutated_oracle_passes_every_pin():
    assert oracle.set_mutation(oracle.MUT_NONE) == oracle.MUT_NONE
    for pin in pins.PINS:
        pin()
