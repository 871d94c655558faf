"""Reader for the small text fixtures in this folder (each cites the page it comes from)."""
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent


def load(name: str) -> dict:
    """Parse ``KEY v v ; v v`` lines into float64 arrays (``;`` separates rows)."""
    out = {}
    for line in (HERE / name).read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        rows = [[float(t) for t in r.split()] for r in rest.split(";")]
        arr = np.array(rows, dtype=np.float64)
        out[key] = arr[0] if arr.shape[0] == 1 and key.startswith(("O_row", "decimals")) else arr
    return out
