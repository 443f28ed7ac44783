"""Failure detection without a GPU fault: a bounded wait that nothing
satisfies gives up after its limit, latches the timeout bit in the context's
status word, and dflash_sync reports DFLASH_ETIMEOUT once; the context stays
usable (a draft afterwards still matches the oracle)."""
import numpy as np
import pytest

import oracle
from synth import TINY, make_weights_np, make_features_np, make_anchor_ids_np
from tests.gpu_util import np_weights_to_device, bf16_dev, i32_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def dfl():
    import __graft_entry__
    __graft_entry__.build()
    import block_diffusion_drafter_pass_gb300 as m
    return m


def test_bounded_wait_reports_timeout_and_context_survives(dfl):
    wn = make_weights_np(TINY, seed=8)
    with dfl.Drafter(TINY, np_weights_to_device(wn, DEV), max_seqs=1, max_batch=1, max_block=8, max_ctx=256,
                     max_fuse_tokens=256) as d:
        d.sync()
        d.debug_wait_timeout(50_000)        # 50 ms
        with pytest.raises(dfl.DFlashError) as e:
            d.sync()
        assert e.value.status == dfl.DFLASH_ETIMEOUT
        d.sync()                            # reported once, then cleared
        with pytest.raises(dfl.DFlashError) as e:
            d.debug_wait_timeout(0)
        assert e.value.status == dfl.DFLASH_EINVAL
        orc = oracle.OracleDrafter(TINY, wn)
        f = make_features_np(40, TINY.n_feat_layers * TINY.hidden, seed=9)
        d.fuse_ctx([0], [40], bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx([0], [40], f, pending=False)
        anchor = make_anchor_ids_np(1, TINY.vocab, seed=10)
        ids = d.draft([0], i32_dev(anchor, DEV), 8).cpu().numpy()[0]
        d.sync()
        ref = orc.draft([0], anchor, 8)[0]
        sure = ref["gap"] > 0.1
        np.testing.assert_array_equal(ids[sure], ref["draft"][sure])
