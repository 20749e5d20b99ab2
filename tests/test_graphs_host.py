"""Host-side logic of the CUDA-graph bucket ladder (no GPU): the device-side
step metadata a replay writes, and the bucket a batch replays."""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def graphs():
    from invariant_fixed_order_gb300 import build
    build.build()
    from invariant_fixed_order_gb300 import graphs as g
    return g


def test_meta_layout_of_a_decode_only_step(graphs):
    """bi_batch.meta for Bk decode rows: [request of token t][position of token t][decode tokens][no prefill
    tokens][logit rows] (the layout include/bi.h documents), padding rows at position 0."""
    pos = np.array([5, 17, 0, 0], np.int32)
    m = graphs.DecodeGraphs._meta(pos, 4)
    assert m.dtype == np.int32 and m.shape == (16,)
    assert m[0:4].tolist() == [0, 1, 2, 3]          # token t belongs to request slot t
    assert m[4:8].tolist() == [5, 17, 0, 0]         # its position
    assert m[8:12].tolist() == [0, 1, 2, 3]         # every token is a decode token, in order
    assert m[12:16].tolist() == [0, 1, 2, 3]        # every row wants logits


def test_bucket_choice(graphs):
    g = object.__new__(graphs.DecodeGraphs)
    g.buckets = {b: None for b in (1, 2, 4, 8, 16, 24)}
    assert [g.bucket_for(b) for b in (1, 2, 3, 5, 9, 17, 24)] == [1, 2, 4, 8, 16, 24, 24]
    with pytest.raises(ValueError):
        g.bucket_for(25)
    assert graphs.LADDER[:6] == (1, 2, 4, 8, 16, 24)   # the page's ladder begins 1, 2, 4, 8, 16, 24
