"""Writes the stored mask picture under tests/golden/ from the oracle alone.

Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def main():
    N, w, s = 32, 8, 4
    mk = oracle.mask(N, w, s)
    lines = [
        "# StreamingLLM attention mask, N = 32 positions, window w = 8 keys of which s = 4 are sinks",
        "# ('#' = attend, '.' = masked; row t = query position, column i = key position).",
        "# Picture of the pattern in page 滑窗与固定稀疏, figure fig-attn-four-mask-compare",
        "# (recent band + sink bar on the left). Written by tests/golden/make_golden.py from the oracle.",
    ]
    lines += ["".join("#" if x else "." for x in row) for row in mk]
    with open(os.path.join(HERE, "streaming_mask_n32_w8_s4.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
