"""Reader for the plain-text fixtures under tests/golden/ ('[name]' headers, rows of tokens)."""
import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name: str, numeric: bool = True) -> dict:
    sections, cur = {}, None
    with open(os.path.join(GOLDEN_DIR, name), encoding="utf-8") as fh:
        for raw in fh:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = line[1:-1]
                sections[cur] = []
                continue
            sections[cur].append(line.split())
    if numeric:
        return {k: np.array([[float(x) for x in row] for row in v]) for k, v in sections.items()}
    return sections
