"""Write parity_example.txt: a bit string and the parity sign after each bit.

Source: "Together AI announces Mamba-3", section 2 (complex-valued states):
the parity task reads a string of 0s and 1s and tracks whether the number of
1s read so far is even or odd.  With A = 0, dt = 1 and an angle of pi on
each 1-bit (0 on each 0-bit), a state started at 1 + 0i has real part +1
after an even count and -1 after an odd count.  The expected signs below
come from counting bits, not from any implementation of the scan.
"""
import os

import numpy as np

bits = np.random.default_rng(2026).integers(0, 2, 48)
signs = ["+" if int(bits[: t + 1].sum()) % 2 == 0 else "-" for t in range(len(bits))]
out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "parity_example.txt")
with open(out, "w") as f:
    f.write("# Parity example; see make_parity_example.py for the source and the rule.\n")
    f.write("bits: " + "".join(str(int(b)) for b in bits) + "\n")
    f.write("signs: " + "".join(signs) + "\n")
