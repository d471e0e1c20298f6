"""Measured parity errors, kept for the record.

Tests call ``record`` with what they measured; when the environment variable
NSM_PARITY_LOG names a file, the session writes every record there as JSON at the end
(tests/conftest.py).  Nothing is written otherwise.
"""

RECORDS = []


def record(name, **values):
    RECORDS.append(dict(name=name, **{k: (float(v) if isinstance(v, (int, float)) else v)
                                      for k, v in values.items()}))
