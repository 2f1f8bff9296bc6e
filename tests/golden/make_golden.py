"""Writes the stored mask picture under tests/golden/ by drawing it from the figure's description, not
from the oracle, so that comparing the oracle's mask against it pins the oracle.

The picture is the StreamingLLM pattern of page 滑窗与固定稀疏 (figure fig-attn-four-mask-compare, its caption
and the StreamingLLM section): every query row t keeps a bar over the first s positions (the sinks) and a
band over its most recent w - s positions, both cut at the diagonal (a key after the query is never
attended).  Drawn here with plain index ranges per row.

Run from the repository root:  python tests/golden/make_golden.py
"""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def draw(N: int, w: int, s: int):
    rows = []
    for t in range(N):
        bar = set(range(0, min(s, t + 1)))              # sinks, left of the diagonal
        band = set(range(max(0, t - (w - s) + 1), t + 1))  # the w - s most recent keys, the row's own included
        rows.append("".join("#" if i in bar or i in band else "." for i in range(N)))
    return rows


def main():
    N, w, s = 32, 8, 4
    lines = [
        "# StreamingLLM attention mask, N = 32 positions, window w = 8 keys of which s = 4 are sinks",
        "# ('#' = attend, '.' = masked; row t = query position, column i = key position).",
        "# Picture of the pattern in page 滑窗与固定稀疏, figure fig-attn-four-mask-compare (recent band +",
        "# sink bar on the left), drawn by tests/golden/make_golden.py from that description with plain",
        "# index ranges per row; the oracle plays no part in writing it.",
    ]
    lines += draw(N, w, s)
    with open(os.path.join(HERE, "streaming_mask_n32_w8_s4.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
