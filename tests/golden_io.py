"""Readers for the text fixtures under tests/golden/ (values printed on the pages)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def worked_example():
    """Returns (routing {token: [experts]}, receive {(rank, expert): [tokens]}, N_a)."""
    route, recv, na = {}, {}, None
    for parts in _lines("worked_example.txt"):
        if parts[0] == "route":
            route[int(parts[1][1:])] = [int(p[1:]) for p in parts[2:]]
        elif parts[0] == "recv":
            recv[(int(parts[1][1:]), int(parts[2][1:]))] = [int(p[1:]) for p in parts[3:]]
        elif parts[0] == "assignments":
            na = int(parts[1])
    return route, recv, na


def scan_example():
    d = {p[0]: [int(v) for v in p[1:]] for p in _lines("scan_example.txt")}
    return d["send_count"], d["send_offset"]


def payload_example():
    return {p[0]: int(p[1]) for p in _lines("payload_88mb.txt")}
