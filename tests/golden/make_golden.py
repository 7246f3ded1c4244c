"""Writes the oracle regression fixtures in this folder.  Calls only ``oracle`` (and the seeded
input generators); nothing here comes from the CUDA path.

The pages print no KDA values for a worked example, so these fixtures are not the pages'
numbers: they freeze the oracle's own results on tiny seeded cases, so that any later change to
the oracle's arithmetic shows up as a failing test and must be justified by a reading of the
pages.  Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
from case_io import gathered_state, gathered_window, oracle_layer  # noqa: E402
from kda_inputs import make_decode, make_verify  # noqa: E402

NAMES = ("q", "k", "v", "f_a", "beta", "gate")


def decode_tiny():
    case = make_decode(seed=21, B=2, H=2, n_steps=3, dk=4, dv=4, r=4, num_slots=3, state_std=0.5,
                       random_conv=True, random_norm=True, random_dt_bias=True)
    L = oracle_layer(case)
    out, S, win = oracle.decode(L, gathered_state(case), gathered_window(case),
                                *(case.inputs[n] for n in NAMES), storage=oracle.STORE_F64)
    return {"case": "make_decode(seed=21, B=2, H=2, n_steps=3, dk=4, dv=4, r=4, num_slots=3, "
                    "state_std=0.5, random_conv, random_norm, random_dt_bias)",
            "out": out.tolist(), "state": S.tolist(), "window": win.tolist()}


def verify_tiny():
    case = make_verify(seed=22, B=2, H=1, T=3, num_slots=4, dk=4, dv=4, r=4, state_std=0.5,
                       random_conv=True)
    L = oracle_layer(case)
    out, rec, recw = oracle.verify(L, gathered_state(case), gathered_window(case),
                                   *(case.inputs[n] for n in NAMES))
    return {"case": "make_verify(seed=22, B=2, H=1, T=3, num_slots=4, dk=4, dv=4, r=4, "
                    "state_std=0.5, random_conv)",
            "out": out.tolist(), "records": rec.tolist(), "window_records": recw.tolist()}


if __name__ == "__main__":
    for name, fn in (("decode_tiny", decode_tiny), ("verify_tiny", verify_tiny)):
        with open(os.path.join(HERE, name + ".json"), "w") as f:
            json.dump(fn(), f, indent=0)
        print("wrote", name)
