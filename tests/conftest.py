import os
import pathlib
import sys

import numpy as np
import pytest

ROOT = pathlib.Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

GOLDEN = pathlib.Path(__file__).resolve().parent / "golden"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled library")
    config.addinivalue_line("markers", "slow: long-running statistical test")


def load_golden(name: str) -> dict:
    """Parse a ``key: v1 v2 ...`` fixture under tests/golden (comments start with #)."""
    out = {}
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split(":", 1)
        out[k.strip()] = v.split()
    return out


def hand_workload(target, draft, ids, gammas=None, *, u=None, E=None, temperature=None, entry="probs",
                  dtype="f32", top_k=None, top_p=None, ncomp=None, slots=None):
    """Assemble a small workload dict by hand (same keys as workloads.make)."""
    target = np.asarray(target, dtype=np.uint16 if dtype == "bf16" else np.float32)
    V = target.shape[-1]
    if draft is not None:
        draft = np.asarray(draft, dtype=np.uint16 if dtype == "bf16" else np.float32)
    ids = np.asarray(ids, dtype=np.int32).reshape(-1)
    T = ids.shape[0]
    N = target.shape[0] - T
    if gammas is None:
        G = T // N if N else 0
        cu = None
    else:
        gammas = np.asarray(gammas, dtype=np.int64)
        G = int(gammas.max()) if len(gammas) else 0
        cu = np.cumsum(gammas).astype(np.int32)
    return dict(entry=entry, dtype=dtype, N=N, gamma=G, V=V, T=T, draft_ids=ids, cu_num_draft_tokens=cu,
                target=target, draft=draft,
                temperature=None if temperature is None else np.asarray(temperature, np.float32),
                top_k=None if top_k is None else np.asarray(top_k, np.int32),
                top_p=None if top_p is None else np.asarray(top_p, np.float32),
                uniforms=None if u is None else np.asarray(u, np.float32).reshape(-1),
                exponentials=None if E is None else np.asarray(E, np.float32).reshape(N, V),
                num_computed_tokens=None if ncomp is None else np.asarray(ncomp, np.int32),
                slot_mapping=None if slots is None else np.asarray(slots, np.int64))


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle
