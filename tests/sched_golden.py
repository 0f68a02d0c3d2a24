"""Reader for the hand-worked scheduler traces in tests/golden/sched_*.txt."""
import glob
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _kv(tokens):
    out = {}
    for t in tokens:
        k, v = t.split("=", 1)
        out[k] = v
    return out


def _ranges(text):
    out = []
    for part in text.split(","):
        a, b = part.split(":")
        out.extend(range(int(a), int(b)))
    return out


def load(path):
    """Returns (config dict, [request dicts], {step: {"seqs": [...], "after": {...}}})."""
    config, requests, steps = None, [], {}
    for raw in open(path):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        tok = line.split()
        if tok[0] == "config":
            config = {k: int(v) for k, v in _kv(tok[1:]).items()}
        elif tok[0] == "request":
            requests.append({k: int(v) for k, v in _kv(tok[1:]).items()})
        elif tok[0] == "step":
            n = int(tok[1])
            st = steps.setdefault(n, {"seqs": [], "after": None, "none": False})
            if tok[2] == "seq":
                kv = _kv(tok[3:])
                st["seqs"].append({"rid": int(kv["rid"]), "q": int(kv["q"]), "ctx": int(kv["ctx"]),
                                   "table": [int(x) for x in kv["table"].split(",")],
                                   "slots": _ranges(kv["slots"])})
            elif tok[2] == "none":
                st["none"] = True
            elif tok[2] == "after":
                st["after"] = {k: int(v) for k, v in _kv(tok[3:]).items()}
    return config, requests, steps


def all_traces():
    return sorted(glob.glob(os.path.join(GOLDEN, "sched_*.txt")))
