"""The seeded generators: a token range drawn on its own equals the same rows
of a longer draw (the chunked run's chunk c is rows 4096c.. of the prompt and
of each layer's logits)."""
import numpy as np

from routing_q4_grouped_gb300 import synth


def test_token_ranges_are_rows_of_the_whole_draw():
    cfg = synth.CONFIGS["chunked"]
    x = synth.gen_x(cfg, 64)
    assert np.array_equal(x[40:56], synth.gen_x(cfg, 16, t0=40))
    lg = synth.gen_logits(cfg, 3, 64)
    assert np.array_equal(lg[50:60], synth.gen_logits(cfg, 3, 10, t0=50))
    for name in ("t4096", "skew"):
        c = synth.CONFIGS[name]
        assert np.array_equal(synth.gen_logits(c, 0, 64)[33:40], synth.gen_logits(c, 0, 7, t0=33))


def test_layers_and_tensors_draw_independent_streams():
    cfg = synth.CONFIGS["chunked"]
    a = synth.gen_logits(cfg, 0, 8)
    b = synth.gen_logits(cfg, 1, 8)
    assert not np.array_equal(a, b)
    assert abs(np.corrcoef(a.ravel(), b.ravel())[0, 1]) < 0.1
