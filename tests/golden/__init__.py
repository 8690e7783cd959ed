"""Parser for the hand-derived fixtures in this folder."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def _num(tok):
    return float.fromhex(tok) if tok.lstrip("-").startswith("0x") else float(tok)


def load_quant_cases(name="quant_tiny.txt"):
    cases, cur = [], None
    with open(os.path.join(HERE, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            toks = rest.split()
            if key == "case":
                cur = {"name": toks[0]}
            elif key == "end":
                cases.append(cur)
                cur = None
            elif key in ("dtype",):
                cur[key] = toks[0]
            elif key in ("bits", "block"):
                cur[key] = int(toks[0])
            elif key in ("x", "y"):
                cur[key] = [_num(t) for t in toks]
            elif key == "codes":
                cur[key] = [int(t) for t in toks]
            elif key in ("packed", "scale_bits"):
                cur[key] = [int(t, 16) for t in toks]
            else:
                raise ValueError(f"unknown key {key!r} in {name}")
    return cases
