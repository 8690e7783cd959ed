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


def load_qgz_case(name="qgz_fused_sum.txt"):
    """A qgZ pipeline case: topology, sizes, sparse inputs and sparse expected values."""
    case = {"x": [], "source_scale_bits": [], "hop1_codes": [], "hop1_scale_bits": [],
            "out_bits": []}
    with open(os.path.join(HERE, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            key, *toks = line.split()
            if key == "topology":
                case["N"], case["M"] = int(toks[0]), int(toks[1])
            elif key in ("bits", "block", "elems_per_rank"):
                case[key] = int(toks[0])
            elif key == "dtype":
                case[key] = toks[0]
            elif key == "x":
                case["x"].append((int(toks[0]), int(toks[1]), _num(toks[2])))
            elif key == "hop1_codes":
                case[key].append((int(toks[0]), int(toks[1]), int(toks[2])))
            elif key in ("source_scale_bits", "hop1_scale_bits", "out_bits"):
                case[key].append((int(toks[0]), int(toks[1]), int(toks[2], 16)))
            else:
                raise ValueError(f"unknown key {key!r} in {name}")
    return case
