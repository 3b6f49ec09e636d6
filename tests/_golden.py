"""Parser for the plan fixtures under tests/golden/ (calls listed per round)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_calls(name):
    names, parent, length = [], [], []
    calls, replay, source = {}, {}, {}
    chunk = None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "chunk":
                chunk = int(tok[1])
            elif tok[0] == "seg":
                names.append(tok[1])
                parent.append(-1 if tok[2] == "-" else names.index(tok[2]))
                length.append(int(tok[3]))
            elif tok[0] == "call":
                rest = " ".join(tok[2:])
                calls[int(tok[1])] = [s.strip().split(",") for s in rest.split("|")]
            elif tok[0] == "replay":
                replay[tok[1]] = int(tok[2])
            elif tok[0] == "source":
                source[tok[1]] = tok[2]
    return dict(names=names, parent=np.array(parent, np.int32),
                seg_len=np.array(length, np.int64), chunk=chunk, calls=calls,
                replay=replay, source=source)


def calls_of(plan, names):
    """Per round, the list of sequences as lists of segment names, in layout order."""
    out = {}
    for r in range(plan["n_rounds"]):
        seqs = []
        for s in range(int(plan["round_seq_ptr"][r]), int(plan["round_seq_ptr"][r + 1])):
            seqs.append([names[v] for v in plan["seq_chain"][s]])
        out[r + 1] = seqs
    return out
