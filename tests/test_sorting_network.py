"""The comparator table of the statistics' shift (csrc/moments.cuh,
shift_of_first8) sorts any 8 values, so its slot 3 is their lower median:
checked on the table as written in the source, by the 0-1 principle (a
comparator network sorts every input if it sorts every 0/1 input) and on
random real values against numpy."""
import itertools
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "diffusion_transformer_qk_gb300", "csrc", "moments.cuh")


def network():
    text = open(SRC).read()
    m = re.search(r"kNet\[(\d+)\]\[2\]\s*=\s*\{(.*?)\};", text, re.S)
    assert m, "comparator table not found"
    pairs = [(int(a), int(b)) for a, b in re.findall(r"\{(\d+),\s*(\d+)\}", m.group(2))]
    assert len(pairs) == int(m.group(1))
    return pairs


def apply(net, values):
    a = list(values)
    for i, j in net:
        a[i], a[j] = min(a[i], a[j]), max(a[i], a[j])
    return a


def test_table_is_well_formed():
    net = network()
    assert len(net) == 19
    assert all(0 <= i < j < 8 for i, j in net)


def test_sorts_every_binary_input():
    net = network()
    for bits in itertools.product((0, 1), repeat=8):
        assert apply(net, bits) == sorted(bits), bits


def test_slot_3_is_the_lower_median_of_real_values():
    net = network()
    g = np.random.Generator(np.random.PCG64(8))
    for row in g.standard_normal((5000, 8)).tolist():
        assert apply(net, row)[3] == sorted(row)[3]
    # ties and an outlier among the first values
    assert apply(net, [3000.0, 1, 1, 2, 0, -1, 1, 5])[3] == 1
