"""End to end through the C ABI: the speculative loop is lossless.

A fake target (a seeded host function of the prefix that agrees with the
drafter's proposal most of the time) stands in for the target model. Each
cycle drafts a block on the GPU, asks the fake target for its greedy ids
after every block position, appends the block's features as pending, and
lets dflash_verify accept and commit. The emitted stream must equal the fake
target's own greedy stream ("DFlash - Block Diffusion for Flash Speculative
Decoding" notes, section 4.5: greedy verification is lossless), and the
library's committed length must track it. Run with plain drafts and with the
path selector installed, for several sequences per call.
"""
import numpy as np
import pytest

from synth import TINY, make_weights_np, make_features_np, make_selector_weights_np
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


class FakeTarget:
    """Greedy next id of a prefix: the proposal with probability p_agree,
    otherwise another id; memoised, so the same prefix always gives the same id."""

    def __init__(self, vocab, seed, p_agree=0.7):
        self.vocab = vocab
        self.rng = np.random.Generator(np.random.PCG64(seed))
        self.p = p_agree
        self.memo = {}

    def next(self, prefix, proposal):
        key = tuple(prefix)
        if key not in self.memo:
            if self.rng.random() < self.p:
                self.memo[key] = int(proposal)
            else:
                self.memo[key] = int((proposal + 1 + self.rng.integers(0, self.vocab - 1)) % self.vocab)
        return self.memo[key]


def _features(seq, pos, width):
    return make_features_np(1, width, seed=100_000 * (seq + 1) + pos)[0]


@pytest.mark.parametrize("selector", [False, True])
def test_speculative_loop_matches_greedy_target(dfl, selector):
    sh = TINY
    wn = make_weights_np(sh, seed=31)
    n, B, target_len = 4, 8, 60
    width = sh.n_feat_layers * sh.hidden
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=n, max_batch=n, max_block=B,
                     max_ctx=target_len + 2 * B + 16, max_fuse_tokens=n * 16) as d:
        if selector:
            sel = make_selector_weights_np(sh, seed=32)
            d.set_path_selector(**{k: bf16_dev(v, DEV) for k, v in sel.items()})
        targets = [FakeTarget(sh.vocab, seed=40 + s) for s in range(n)]
        prompts = [[11 + s, 12, 13 + 2 * s, 14, 15][: 3 + s % 3] for s in range(n)]
        seqs = list(range(n))
        feats = np.concatenate([np.stack([_features(s, i, width) for i in range(len(prompts[s]))]) for s in seqs])
        d.fuse_ctx(seqs, [len(p) for p in prompts], bf16_dev(feats, DEV), pending=False)
        outs = [list(p) for p in prompts]
        anchors = []
        for s in seqs:
            outs[s].append(targets[s].next(outs[s], 0))
            anchors.append(outs[s][-1])
        taus = []
        while max(len(o) for o in outs) < target_len:
            drafts = d.draft(seqs, i32_dev(anchors, DEV), B).cpu().numpy()
            t_ids = np.zeros((n, B), dtype=np.int32)
            fb = []
            for s in seqs:
                block = [anchors[s]] + [int(x) for x in drafts[s]]
                prefix = outs[s][:-1]
                for j in range(B):
                    prop = block[j + 1] if j + 1 < B else 0
                    t_ids[s, j] = targets[s].next(prefix + block[: j + 1], prop)
                fb.append(np.stack([_features(s, len(prefix) + j + 1, width) for j in range(B)]))
            d.fuse_ctx(seqs, [B] * n, bf16_dev(np.concatenate(fb), DEV), pending=True)
            tau, bonus = d.verify(seqs, B, i32_dev(drafts, DEV), i32_dev(t_ids, DEV))
            tau, bonus = tau.cpu().numpy(), bonus.cpu().numpy()
            for s in seqs:
                block = [anchors[s]] + [int(x) for x in drafts[s]]
                outs[s] += block[1:int(tau[s])] + [int(bonus[s])]
                anchors[s] = int(bonus[s])
                taus.append(int(tau[s]))
                assert d.seq_len(s) == (len(outs[s]) - 1, 0)
        for s in seqs:
            greedy = list(prompts[s])
            while len(greedy) < len(outs[s]):
                greedy.append(targets[s].memo[tuple(greedy)])
            assert greedy == outs[s], f"sequence {s}"
        assert max(taus) > 1 and min(taus) >= 1
