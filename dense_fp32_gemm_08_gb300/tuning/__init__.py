"""Per-shape-class configuration tuning: `sweep.py` measures, `gen_table.py` writes the table."""
