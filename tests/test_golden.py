"""Values the pages print, stored under tests/golden/ with their citations, against the oracle
and against the library's host metadata call (no GPU needed)."""
import json
import os

import numpy as np
import pytest

import selective_state_space_mamba2_gb300 as ssd

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _cases(name):
    with open(os.path.join(GOLDEN, name)) as f:
        doc = json.load(f)
    assert doc["citation"]
    return doc["cases"]


WARMUP = _cases("warmup_chunk_metadata.json")
KEYS = ("cu_chunk_seqlens", "seq_idx", "last_chunk_indices")


@pytest.mark.parametrize("case", WARMUP, ids=lambda c: "Q%d" % c["chunk_size"])
def test_warmup_metadata_oracle(oracle_lib, case):
    m = oracle_lib.chunk_metadata(case["cu_seqlens"], case["num_computed_tokens"], case["chunk_size"])
    for k in KEYS:
        assert m[k].tolist() == case[k], k


@pytest.mark.parametrize("case", WARMUP, ids=lambda c: "Q%d" % c["chunk_size"])
def test_warmup_metadata_library(case):
    ssd.build()
    m = ssd.ssd_chunk_metadata(np.array(case["cu_seqlens"], np.int32), case["chunk_size"],
                               np.array(case["num_computed_tokens"], np.int32))
    for k in KEYS:
        assert m[k].tolist() == case[k], k
