"""Write tests/golden/screened_attempts.json: for every parity workload, the
attempt number of a draw of each sequence that clears the decision margins
of tests/parity.py (the search starts from the table's previous entry, if
any).  Calls only the seeded generator and the oracle; the tests re-check
every stored draw and redraw themselves if one fails, so the table only
saves the search.

    python tests/golden/make_screened_attempts.py [workload ...]
"""
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import synth  # noqa: E402
from parity import GOLDEN_ATTEMPTS, order_margins, screen  # noqa: E402

# the workloads the GPU parity tests screen: the pages' five (six with the
# late phase) and the literal reading of the logit boost on the two small ones
WORKLOADS = [(n, "relative") for n in synth.ORDER] + [("tiny", "absolute"), ("llada_step", "absolute")]


def main(names):
    table = {}
    if os.path.exists(GOLDEN_ATTEMPTS):
        with open(GOLDEN_ATTEMPTS) as fh:
            table = json.load(fh)
    for name, mode in WORKLOADS:
        if names and name not in names and f"{name}:{mode}" not in names:
            continue
        cfg = synth.scaled(synth.CONFIGS[name], boost_mode=mode)
        seed = 1000 + synth.ORDER.index(name)
        t0 = time.time()
        log = []
        key = f"{name}:{mode}:{seed}"
        start = table.get(key, {}).get("attempts")   # a search under other margins resumes from its draws
        w, _ = screen(cfg, seed, attempts=start, use_stored=False, log=log)
        table[key] = dict(order_margins=order_margins(cfg), attempts=[int(a) for a in w.attempts])
        print(f"{name}:{mode} seed {seed}: {len(log)} redraws, max attempt {int(w.attempts.max())}, "
              f"{time.time() - t0:.0f} s", flush=True)
    with open(GOLDEN_ATTEMPTS, "w") as fh:
        json.dump(table, fh, indent=1, sort_keys=True)
        fh.write("\n")


if __name__ == "__main__":
    main(sys.argv[1:])
