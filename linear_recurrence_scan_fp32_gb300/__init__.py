"""GB300-native first-order linear-recurrence scan (binding filled in below)."""
