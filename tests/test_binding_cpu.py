"""Host-side marshalling of the Python binding (no GPU): the byte layout pack_layer builds
for layer streaming."""
import numpy as np
import pytest

import synth
from bit_weight_quantized_dequant_gb300 import FMT_2BIT, FMT_NF4, pack_layer
from oracle import oracle as O

SHAPES = [(48, 256), (16, 512), (40, 1024)]


@pytest.mark.parametrize("fmt", [FMT_2BIT, FMT_NF4])
def test_pack_layer_places_every_array_at_its_offset(fmt):
    if fmt == FMT_2BIT:
        packs = [synth.random_packed_2bit(N, K, O.anchor_count(K), seed=2, matrix_id=i) for i, (N, K) in enumerate(SHAPES)]
        fields = [("codes", "codes"), ("scales", "scales"), ("offsets", "offsets"), ("anchor_idx", "anchor_idx"),
                  ("anchor_w", "anchor_w")]
    else:
        packs = [synth.random_packed_nf4(N, K, seed=2, matrix_id=i) for i, (N, K) in enumerate(SHAPES)]
        fields = [("codes", "codes"), ("scales", "absmax")]
    blob, meta = pack_layer(packs, fmt)
    assert blob.dtype == np.uint8 and blob.nbytes % 256 == 0
    starts = []
    for p, m in zip(packs, meta):
        assert (m["N"], m["K"]) == (p["N"], p["K"])
        for key, src in fields:
            a = np.ascontiguousarray(p[src]).view(np.uint8).reshape(-1)
            off = m[key]
            assert off % 256 == 0
            assert np.array_equal(blob[off:off + a.nbytes], a), key
            starts.append((off, off + a.nbytes))
        if fmt == FMT_2BIT:
            assert m["A"] == p["A"] and m["ld_anchor"] == p["ld_anchor"]
        else:
            assert m["offsets"] == m["anchor_idx"] == m["anchor_w"] == 0 and m["A"] == 0
    starts.sort()
    for (a0, a1), (b0, _) in zip(starts, starts[1:]):
        assert a1 <= b0                                  # no two arrays overlap
    assert starts[-1][1] <= blob.nbytes
