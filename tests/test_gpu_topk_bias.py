"""Top-K parity on logits that rise along the vocabulary.

The lm_head kernel keeps, in every CTA, a sorted list of the K best logits of
each position and filters each new vocabulary tile against per-position
thresholds. From a CTA's third tile on, the survivors are filed into
fixed-size per-position buckets; a tile in which some position has more
survivors than its bucket holds is processed again by the chunked path. With
the workloads' random weights the buckets rarely fill.

Here every vocabulary row gets a bias that grows with its tile index (hidden
component 0 is 1 and weight column 0 holds the bias), so each new tile of a
CTA beats many of the logits it has kept: buckets overflow in many tiles and
CTAs, next to tiles whose survivors fit. The whole selector must still match
the oracle under the usual parity rules.
"""
import pytest
import torch

from tests import parity
from speculative_decoding_draft_tcgen05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_draft_tcgen05_gb300 import build
    build.build()
    import speculative_decoding_draft_tcgen05_gb300 as p
    p.lib()
    return p


def rising_inputs(w, step):
    """The workload's inputs with U_t(v) raised by step * (v // 128)."""
    inp = wl.make_inputs(w)
    tile = torch.div(torch.arange(w.V), 128, rounding_mode="floor").to(torch.float32)
    inp.W[:, 0] = (tile * step).to(torch.bfloat16)
    inp.hidden[..., 0] = 1.0
    return inp


# V = 65536 gives each lm_head CTA three or more tiles. The bias step per tile
# is chosen so that a CTA's next tile sits about three logit standard
# deviations (0.05 * sqrt(127)) above its previous one.
CASES = [
    # 224 positions: two position tiles of 112, buckets of 9 keys per position
    (wl.custom(name="rising_b32", B=32, L=7, K=16, V=65536, d=128, seed=31, std_w=0.05), 0.022),
    # 56 positions: one position tile of 64, buckets of 16 keys per position
    (wl.custom(name="rising_b8", B=8, L=7, K=16, V=65536, d=128, seed=32, std_w=0.05), 0.012),
    # K = 32 on a 32-wide position tile (buckets of 32 keys): the per-tile path's
    # 32-entry insertion; V = 50000 gives 89 CTAs a third tile
    (wl.custom(name="rising_k32", B=4, L=8, K=32, V=50000, d=128, seed=33, std_w=0.05), 0.012),
]


@pytest.mark.parametrize("w,step", CASES, ids=[c[0].name for c in CASES])
def test_rising_logits_match_oracle(pkg, w, step):
    inp = rising_inputs(w, step)
    gpu = parity.run_gpu(inp)
    orc = parity.run_oracle(inp, range(w.B))
    rep = parity.compare(inp, gpu, orc)
    assert rep["positions"] == w.B * w.L
    # most positions are compared exactly: the bias packs many logits near the
    # K-th one, so some top-K margins fall below the tie threshold (6 of 56 at
    # rising_b8), but not most
    assert rep["topk_excused"] <= w.B * w.L // 4, rep
