"""KV block manager: the oracle's pins (CPU only)."""
import pytest

from oracle.block_manager import BlockManager, OutOfBlocks
from tests import bm_checks as bc


def oracle_factory(mutation=0):
    return lambda nb, B, order: BlockManager(nb, B, free_order=order, mutation=mutation)


@pytest.mark.parametrize("check", bc.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle_factory())


MUTANTS = {1: "copy keeps the shared count", 2: "shared block written in place",
           3: "offset off by one", 4: "freed blocks lost", 5: "fork not counted"}


@pytest.mark.parametrize("mutation", sorted(MUTANTS), ids=lambda m: MUTANTS[m])
def test_oracle_planted_mistake_is_caught(mutation):
    caught = []
    for check in bc.ALL_CHECKS:
        try:
            check(oracle_factory(mutation))
        except (AssertionError, OutOfBlocks, IndexError, KeyError):
            caught.append(check.__name__)
    assert caught, f"mutation {MUTANTS[mutation]} passed every pin"


def test_oracle_rejects_bad_calls():
    bm = BlockManager(8, 4)
    bm.add(1)
    with pytest.raises(KeyError):
        bm.add(1)
    with pytest.raises(KeyError):
        bm.append(2, 1)
    with pytest.raises(KeyError):
        bm.fork(2, 3)
    with pytest.raises(ValueError):
        bm.append_batch([1, 1], [1, 1])
    with pytest.raises(ValueError):
        bm.append(1, -1)
    with pytest.raises(ValueError):
        BlockManager(4, 4, free_order=[0, 1, 2, 2])
