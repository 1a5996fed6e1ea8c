"""Format the per-case records of the stress-sweep parity tests (the JSON
lines the GPU tests append when FA_PARITY_REPORT is set) as the markdown
report beside this file:

    FA_PARITY_REPORT=parity_report.jsonl python -m pytest tests -m gpu -q
    python tests/reports/make_stress_report.py parity_report.jsonl > tests/reports/stress_parity_C5.md
"""
import json, sys, math
rows=[json.loads(l) for l in open(sys.argv[1])]
fw=[r for r in rows if r['dir']=='fwd']; bw=[r for r in rows if r['dir']=='bwd']
def key(c):
    p=c.split('_'); return (int(p[3][1:]), int(p[2][1:]), p[4])
agg={}
for r in fw:
    a=agg.setdefault(r['case'],dict(o=0,oref=0,v=0,over=0,n=0,lse=0))
    a['o']=max(a['o'],r['o_max_err']); a['oref']=max(a['oref'],r['o_ref_max_abs']); a['v']=max(a['v'],r['v_max_abs']); a['over']+=r['over_plain_gate']; a['n']+=r['elements']; a['lse']=max(a['lse'],r['lse_max_err'])
out=[]
out.append("# Stress-sweep parity report (C5: D in {64, 128, 256}, S in {1024, 4096, 16384}, B*S = 16384, H = 16)\n")
out.append("Inputs: Q ~ N(0, 4^2), K ~ N(0, 1) with 1 % of key rows x8 per head, V, dO ~ N(0, 1), bf16, seed 0, scale 1/sqrt(D). Checked heads (0, 0) and (B-1, 15); S = 16384 on 128 sampled rows (and key columns), all rows otherwise. Oracle: the fp64 CPU reference in `oracle/`.\n")
out.append("Written by the GPU parity tests `tests/test_fwd_gpu.py::test_stress_sweep` and `tests/test_bwd_gpu.py::test_stress_sweep` on a GB300, with the per-case records they append when `FA_PARITY_REPORT` is set:\n")
out.append("```\nFA_PARITY_REPORT=parity_report.jsonl python -m pytest tests -m gpu -q\npython tests/reports/make_stress_report.py parity_report.jsonl > tests/reports/stress_parity_C5.md\n```\n")
out.append("## Forward\n")
out.append("Gates: LSE max-abs <= 1e-3; O max-abs <= 1e-2 + ulp_bf16(O_ref)/2 (the plain gate) plus, for these peaked inputs, 2^-9 max|V| (the bound on what the bf16 rounding of P can move O by), with at most 1e-5 of the elements above the plain gate.\n")
out.append("| case | max abs O error | max abs O_ref | max abs V | 2^-9 max abs V | elements above the plain gate | elements checked | max abs LSE error |")
out.append("|---|---|---|---|---|---|---|---|")
for c in sorted(agg, key=key):
    a=agg[c]
    out.append(f"| {c} | {a['o']:.4f} | {a['oref']:.3f} | {a['v']:.3f} | {a['v']/512:.4f} | {a['over']} | {a['n']} | {a['lse']:.2e} |")
out.append("\n## Backward\n")
out.append("Gate: relative L2 error <= 2e-2 per tensor over the checked heads (rows / key columns).\n")
out.append("| case | dQ rel L2 | dK rel L2 | dV rel L2 |")
out.append("|---|---|---|---|")
for r in sorted(bw, key=lambda r: key(r['case'])):
    out.append(f"| {r['case']} | {r['dq_rel_l2']:.4f} | {r['dk_rel_l2']:.4f} | {r['dv_rel_l2']:.4f} |")
mo=max(a['o'] for a in agg.values()); tot=sum(a['over'] for a in agg.values()); n=sum(a['n'] for a in agg.values())
out.append(f"\nLargest O error over the 18 cases: {mo:.4f}; {tot} of {n} checked O elements exceed the plain gate, all within the P-rounding allowance. Largest gradient error: {max(max(r['dq_rel_l2'],r['dk_rel_l2'],r['dv_rel_l2']) for r in bw):.4f}.")
print("\n".join(out))
