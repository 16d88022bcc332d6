"""Memory utilisation, contiguous reservation vs paging, on a continuous batch
(host simulation through the library's block manager).  The block counts are
checked at every step against the oracle's closed-form accounting; the
outcome is checked against the pages' claims: a sequence wastes less than one
block with paging (utilisation above 96 %), while reserving the maximum length
leaves most of the memory unused and admits several times fewer requests."""
import pytest

from oracle import accounting
from paged_kv_cache_237_gb300 import build as pa_build


@pytest.fixture(scope="module")
def sim():
    pa_build.build()
    from paged_kv_cache_237_gb300 import memory_sim
    return memory_sim


@pytest.mark.parametrize("block_size", [16, 32])
def test_paged_vs_contiguous_utilisation(sim, block_size):
    max_len = 32768
    prompts, outputs = sim.request_stream(120, seed=3, max_len=max_len)
    budget = 40 * max_len                     # room for 40 maximum-length reservations

    def check(bm, running):
        held_blocks = accounting.shared_prefix_blocks(0, list(running.values()), block_size)
        assert bm.num_free() == budget // block_size - held_blocks
        assert accounting.paged_slack_tokens(list(running.values()), block_size) < block_size * max(1, len(running))

    paged = sim.simulate_paged(prompts, outputs, budget, block_size, check=check)
    contig = sim.simulate_contiguous(prompts, outputs, budget, max_len)
    assert paged.finished == contig.finished == 120
    assert paged.mean_utilisation > 0.96
    assert contig.mean_utilisation < 0.6
    assert paged.mean_running > 2.0 * contig.mean_running
    assert paged.steps < contig.steps
