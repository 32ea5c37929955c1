"""Write closed_form_decode.json: decode results derived by hand.

Uses only the closed form of softmax attention (no oracle, no library), so the
stored values pin the oracle to mathematics rather than to itself:
  s_j = scale * (q . row_j);  lse = ln sum_j exp(s_j);
  o   = sum_j exp(s_j - lse) * row_j[0:kv_rank].
Run: python tests/golden/make_closed_forms.py
"""
import json
import math
import os

cases = []

# two keys, kv_rank 2, no rope: q = e_0, rows = e_0, e_1, scale 1
# s = [1, 0]; lse = ln(e + 1); o = [e/(e+1), 1/(e+1)]
e = math.e
cases.append({"name": "two_keys", "kv_rank": 2, "block_size": 16, "scale": 1.0,
              "q": [1.0, 0.0], "rows": [[1.0, 0.0], [0.0, 1.0]],
              "o": [e / (e + 1), 1 / (e + 1)], "lse": math.log(e + 1)})

# rope column decides the scores: kv_rank 1, d_rope 1, q = [0, 2]
# rows [3, 0.5], [5, -0.5]: s = [1, -1]; lse = ln(e + 1/e) = ln(2 cosh 1)
# o = (3 e + 5/e) / (e + 1/e)
cases.append({"name": "rope_tail", "kv_rank": 1, "block_size": 16, "scale": 1.0,
              "q": [0.0, 2.0], "rows": [[3.0, 0.5], [5.0, -0.5]],
              "o": [(3 * e + 5 / e) / (e + 1 / e)], "lse": math.log(2 * math.cosh(1.0))})

# 18 keys across a block boundary (block size 16); key j = [j, 1], q = [0, 1],
# scale 1: every score is 1 so the weights are uniform;
# o = mean(j) = 8.5, lse = 1 + ln 18
rows = [[float(j), 1.0] for j in range(18)]
cases.append({"name": "uniform_across_blocks", "kv_rank": 1, "block_size": 16,
              "scale": 1.0, "q": [0.0, 1.0], "rows": rows, "o": [8.5],
              "lse": 1.0 + math.log(18.0)})

# scale 0.5, keys [2, 0] and [0, 0] with q = [1, 0] (kv_rank 2):
# s = [1, 0] again; o = [2 e/(e+1), 0]
cases.append({"name": "scaled", "kv_rank": 2, "block_size": 16, "scale": 0.5,
              "q": [1.0, 0.0], "rows": [[2.0, 0.0], [0.0, 0.0]],
              "o": [2 * e / (e + 1), 0.0], "lse": math.log(e + 1)})

out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_form_decode.json")
with open(out, "w") as f:
    json.dump({"about": "hand-derived absorbed-decode results (see make_closed_forms.py)",
               "cases": cases}, f, indent=1)
print("wrote", out)
