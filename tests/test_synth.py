"""The stored routing counts of the synthetic workloads re-derive from their seeds."""

import synth


def test_routing_counts_rederive_from_seeds():
    c3, c4, c5 = synth.routing_counts_from_seed()
    assert c3 == synth.COUNTS_CONTIG and sum(c3) == 16384
    assert c4 == synth.MASKED_M and sum(c4) == 10002
    assert c5 == synth.UNITS_DSWIGLU and sum(c5) == 128


def test_padded_offsets():
    off = synth.padded_offsets_from_counts(synth.COUNTS_CONTIG)
    assert off.tolist() == [256, 5888, 6144, 10240, 11264, 12544, 16896, 17408]
    assert synth.padded_offsets_from_counts([0, 1, 256]).tolist() == [0, 256, 512]
